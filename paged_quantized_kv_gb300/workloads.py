"""Seeded synthetic workloads for the NVFP4 KV store and the indexer-K gather.

This module only draws inputs (numpy ``default_rng``); it holds none of the
quantisation or gather arithmetic, so the CUDA path and the CPU oracle can
both consume its arrays.  Every array is produced on the host as exact
bytes; callers copy them to the device.

Named workloads (seed = workload index unless given):

0. ``tiny`` -- store: 24 tokens, 2 KV heads, head_size 64, block_size 16,
   8-block cache, bf16 N(0,1) with one x20 outlier per (side, head),
   k_scale = v_scale = 1, 24 distinct random slots in [0, 128) with 3 set
   to -1.  Gather: sequences of 5 and 37 tokens, block_size 64, head_dim 128,
   4-block cache, random non-NaN e4m3 K bytes, scales U[1e-3, 1], block table
   a random permutation of the 4 blocks as [2, 2].
1. ``decode`` -- store: 256 tokens (one per request), 8 heads, head_size 128,
   block_size 16, N(0,1), per-tensor scale amax/(448*6), 65536-block cache,
   256 random distinct slots.
2. ``prefill`` -- store: 16 requests x 1024 tokens, 8 heads, head_size 128,
   block_size 16, N(0,1) with 0.1% of values x50, per-tensor scales, each
   request's tokens in contiguous runs over 64 randomly chosen blocks of a
   65536-block cache; K and V are the two halves of a [T, 2, H, D] buffer
   (row stride 2*H*D).
3. ``prefill_gather`` -- gather: 16 sequences with lengths U[1000, 8192],
   block_size 64, head_dim 128, 4096-block cache, log-uniform scales in
   [1e-4, 1], block table [16, 128] from a random permutation of the blocks.
4. ``long`` -- (a) store: 256 requests x 512 tokens, 4 heads, head_size 256,
   block_size 32, N(0,1), per-tensor scales, each request on 16 blocks of a
   4096-block cache in random order; (b) gather: 256 sequences x 512 tokens,
   block_size 64, head_dim 128, 8192-block cache, block table [256, 8].
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

LAYOUT_HND = 0
LAYOUT_NHD = 1
DTYPE_BF16 = 0
DTYPE_F16 = 1


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even, torch's CPU cast) as uint16."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> exact fp32 values."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> IEEE fp16 (round to nearest even, numpy's cast) as uint16."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(
        np.float16).view(np.uint16)


def element_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    return f16_bits(x) if dtype == DTYPE_F16 else bf16_bits(x)


def element_values(bits: np.ndarray, dtype: int) -> np.ndarray:
    """uint16 bit patterns of the given element type -> fp32 values."""
    if dtype == DTYPE_F16:
        return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(
            np.float32)
    return bf16_values(np.asarray(bits))


@dataclass
class StoreWorkload:
    """Inputs of one NVFP4 paged store.

    ``src`` is the flat bf16 (uint16 bits) backing buffer; key token t, head
    h, element d sits at ``key_offset + t*key_stride0 + h*D + d`` and value
    likewise.  The cache is ``num_blocks`` pages of ``page_stride`` bytes;
    the K side of a page starts at byte 0 of the page and the V side at
    ``value_side_offset``."""
    name: str
    num_tokens: int
    num_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    src: np.ndarray
    key_offset: int
    key_stride0: int
    value_offset: int
    value_stride0: int
    slot_mapping: np.ndarray
    k_scale: np.float32
    v_scale: np.float32
    layout: int = LAYOUT_HND
    flags: int = 0
    page_stride: int = 0
    dtype: int = DTYPE_BF16
    extra: dict = field(default_factory=dict)

    def __post_init__(self):
        if self.page_stride == 0:
            self.page_stride = 2 * self.side_bytes

    @property
    def scale_dim(self) -> int:
        return self.head_size // 16

    @property
    def side_bytes(self) -> int:
        H, B, D = self.num_heads, self.block_size, self.head_size
        return H * B * (D // 2 + D // 16)

    @property
    def value_side_offset(self) -> int:
        return self.side_bytes

    @property
    def cache_bytes(self) -> int:
        return self.num_blocks * self.page_stride

    @property
    def stored_tokens(self) -> int:
        return int((self.slot_mapping[: self.num_tokens] >= 0).sum())

    def algorithmic_bytes(self) -> int:
        """bf16 K and V read + int64 slot read + NVFP4 data and scales
        written, for the tokens that are stored (a skipped token reads only
        its slot)."""
        H, D = self.num_heads, self.head_size
        n = self.stored_tokens
        return (n * 2 * H * D * 2 + self.num_tokens * 8
                + n * 2 * H * (D // 2 + D // 16))

    def key_array(self) -> np.ndarray:
        """[T, H, D] view of the key bits (strided)."""
        return _view(self.src, self.key_offset, self.key_stride0,
                     self.num_tokens, self.num_heads, self.head_size)

    def value_array(self) -> np.ndarray:
        return _view(self.src, self.value_offset, self.value_stride0,
                     self.num_tokens, self.num_heads, self.head_size)


def _view(src, offset, stride0, T, H, D):
    if T == 0:
        return np.zeros((0, H, D), dtype=np.uint16)
    it = src.itemsize
    return np.lib.stride_tricks.as_strided(
        src[offset:], shape=(T, H, D), strides=(stride0 * it, D * it, it),
        writeable=False)


@dataclass
class GatherWorkload:
    """Inputs of one indexer-K gather.

    ``cache`` holds ``num_blocks`` blocks of ``block_stride`` bytes; block =
    [block_size*head_dim fp8 K | block_size*4 fp32 scale bytes]."""
    name: str
    block_size: int
    head_dim: int
    num_blocks: int
    cache: np.ndarray
    block_table: np.ndarray
    cu_seq_lens: np.ndarray
    block_stride: int = 0
    extra: dict = field(default_factory=dict)

    def __post_init__(self):
        if self.block_stride == 0:
            self.block_stride = self.block_size * (self.head_dim + 4)

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seq_lens.size - 1)

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seq_lens[-1])

    def algorithmic_bytes(self) -> int:
        """K row and scale read and written per token, plus the block-table
        entries and cu_seq_lens read."""
        B = self.block_size
        lens = np.diff(self.cu_seq_lens.astype(np.int64))
        table_entries = int(((lens + B - 1) // B).sum())
        return (self.total_tokens * 2 * (self.head_dim + 4)
                + 4 * table_entries + 4 * self.cu_seq_lens.size)


# --- generators ---------------------------------------------------------------

def random_e4m3_bytes(rng, n: int) -> np.ndarray:
    """n bytes uniform over the 254 non-NaN e4m3 codes (all but 0x7F, 0xFF)."""
    v = rng.integers(0, 254, size=n, dtype=np.int32)
    v = np.where(v >= 0x7F, v + 1, v)
    return v.astype(np.uint8)


def _normal_f32(rng, shape, outlier_p=0.0, outlier_mult=1.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if outlier_p > 0:
        mask = rng.random(size=shape) < outlier_p
        x = np.where(mask, x * np.float32(outlier_mult), x)
    return x


def per_tensor_scale(bits: np.ndarray, dtype: int = DTYPE_BF16) -> np.float32:
    """Checkpoint scale recipe of the decode/prefill workloads:
    amax(|x|) / (448 * 6) in fp32."""
    if bits.size == 0:
        return np.float32(1.0)
    amax = np.abs(element_values(bits, dtype)).max()
    return np.float32(amax) / np.float32(448.0 * 6.0)


def make_store(name: str, seed: int, num_tokens: int, num_heads: int,
               head_size: int, block_size: int, num_blocks: int,
               slots: str = "random", skip: int = 0, row_mult: int = 1,
               outlier_p: float = 0.0, outlier_mult: float = 1.0,
               outlier_per_head: float = 0.0, scales: str = "per_tensor",
               request_len: int = 0, layout: int = LAYOUT_HND,
               flags: int = 0, dtype: int = DTYPE_BF16) -> StoreWorkload:
    """Generic store workload.

    slots: "random" (distinct random slots over the whole cache),
    "runs" (requests of ``request_len`` tokens, each on randomly chosen
    distinct blocks filled in order), or "dense" (token t -> slot t).
    skip: number of tokens whose slot is set to -1.
    row_mult: K and V are halves of a [T, row_mult, H, D] buffer when 2.
    dtype: element type of K and V (bf16 or fp16 bit patterns)."""
    rng = np.random.default_rng(seed)
    T, H, D, B = num_tokens, num_heads, head_size, block_size
    if row_mult == 2:
        x = _normal_f32(rng, (T, 2, H, D), outlier_p, outlier_mult)
        if outlier_per_head:
            for side in range(2):
                for h in range(H):
                    t = rng.integers(0, max(T, 1))
                    d = rng.integers(0, D)
                    if T:
                        x[t, side, h, d] *= np.float32(outlier_per_head)
        src = element_bits(x.reshape(-1), dtype)
        key_offset, value_offset, stride0 = 0, H * D, 2 * H * D
    else:
        kx = _normal_f32(rng, (T, H, D), outlier_p, outlier_mult)
        vx = _normal_f32(rng, (T, H, D), outlier_p, outlier_mult)
        if outlier_per_head and T:
            for arr in (kx, vx):
                for h in range(H):
                    t = rng.integers(0, T)
                    d = rng.integers(0, D)
                    arr[t, h, d] *= np.float32(outlier_per_head)
        src = element_bits(np.concatenate([kx.reshape(-1), vx.reshape(-1)]),
                           dtype)
        key_offset, value_offset, stride0 = 0, T * H * D, H * D

    capacity = num_blocks * B
    if slots == "random":
        sm = rng.choice(capacity, size=T, replace=False).astype(np.int64)
    elif slots == "dense":
        sm = np.arange(T, dtype=np.int64)
    elif slots == "runs":
        assert request_len > 0 and T % request_len == 0
        n_req = T // request_len
        bpr = (request_len + B - 1) // B
        blocks = rng.permutation(num_blocks)[: n_req * bpr].reshape(n_req, bpr)
        k = np.arange(request_len)
        sm = (blocks[:, k // B] * B + (k % B)[None, :]).reshape(-1)
        sm = sm.astype(np.int64)
    else:
        raise ValueError(slots)
    if skip:
        sm[rng.choice(T, size=skip, replace=False)] = -1

    wl = StoreWorkload(name=name, num_tokens=T, num_heads=H, head_size=D,
                       block_size=B, num_blocks=num_blocks, src=src,
                       key_offset=key_offset, key_stride0=stride0,
                       value_offset=value_offset, value_stride0=stride0,
                       slot_mapping=sm, k_scale=np.float32(1.0),
                       v_scale=np.float32(1.0), layout=layout, flags=flags,
                       dtype=dtype)
    if scales == "per_tensor":
        wl.k_scale = per_tensor_scale(np.asarray(wl.key_array()), dtype)
        wl.v_scale = per_tensor_scale(np.asarray(wl.value_array()), dtype)
    elif scales == "one":
        pass
    else:
        wl.k_scale, wl.v_scale = np.float32(scales[0]), np.float32(scales[1])
    return wl


def make_gather(name: str, seed: int, seq_lens, block_size: int,
                head_dim: int, num_blocks: int, max_blocks: int = 0,
                scales: str = "log", block_stride: int = 0) -> GatherWorkload:
    """Generic gather workload: random non-NaN e4m3 K bytes, fp32 scales
    ("uniform": U[1e-3, 1]; "log": 10^U(-4, 0)), block table rows filled
    from one random permutation of the cache's blocks."""
    rng = np.random.default_rng(seed)
    B, D = block_size, head_dim
    stride = block_stride or B * (D + 4)
    lens = np.asarray(seq_lens, dtype=np.int64)
    n = lens.size
    need = (lens + B - 1) // B
    mb = max_blocks or max(int(need.max()) if n else 1, 1)
    cache = np.zeros((num_blocks, stride), dtype=np.uint8)
    cache[:, : B * D] = random_e4m3_bytes(rng, num_blocks * B * D).reshape(
        num_blocks, B * D)
    if scales == "uniform":
        sc = rng.uniform(1e-3, 1.0, size=(num_blocks, B)).astype(np.float32)
    else:
        sc = (10.0 ** rng.uniform(-4.0, 0.0, size=(num_blocks, B))).astype(
            np.float32)
    cache[:, B * D: B * D + 4 * B] = sc.view(np.uint8).reshape(num_blocks,
                                                               4 * B)
    perm = rng.permutation(num_blocks).astype(np.int32)
    assert n * mb <= num_blocks
    block_table = perm[: n * mb].reshape(n, mb).copy()
    cu = np.zeros(n + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    return GatherWorkload(name=name, block_size=B, head_dim=D,
                          num_blocks=num_blocks, cache=cache.reshape(-1),
                          block_table=block_table, cu_seq_lens=cu,
                          block_stride=stride)


# --- the five named workloads --------------------------------------------------

def store_workload(index: int, seed: int | None = None) -> StoreWorkload:
    s = index if seed is None else seed
    if index == 0:
        return make_store("tiny_store", s, 24, 2, 64, 16, 8, slots="random",
                          skip=3, outlier_per_head=20.0, scales="one")
    if index == 1:
        return make_store("decode_store", s, 256, 8, 128, 16, 65536,
                          slots="random")
    if index == 2:
        return make_store("prefill_store", s, 16384, 8, 128, 16, 65536,
                          slots="runs", request_len=1024, row_mult=2,
                          outlier_p=1e-3, outlier_mult=50.0)
    if index == 4:
        return make_store("long_store", s, 131072, 4, 256, 32, 4096,
                          slots="runs", request_len=512)
    raise ValueError(f"workload {index} has no store part")


def gather_workload(index: int, seed: int | None = None) -> GatherWorkload:
    s = index if seed is None else seed
    if index == 0:
        return make_gather("tiny_gather", s, [5, 37], 64, 128, 4,
                           max_blocks=2, scales="uniform")
    if index == 3:
        lens = np.random.default_rng([s, 1]).integers(1000, 8192, size=16,
                                                       endpoint=True)
        return make_gather("prefill_gather", s, lens, 64, 128, 4096,
                           max_blocks=128)
    if index == 4:
        return make_gather("long_gather", s, [512] * 256, 64, 128, 8192,
                           max_blocks=8)
    raise ValueError(f"workload {index} has no gather part")


# --- sharding across ranks (data parallel, no exchange) ----------------------------

def shard_range(n: int, rank: int, world: int):
    """Contiguous [lo, hi) share of n units for one rank."""
    lo = (n * rank) // world
    hi = (n * (rank + 1)) // world
    return lo, hi


def shard_store(wl: StoreWorkload, rank: int, world: int,
                unit_tokens: int = 1) -> StoreWorkload:
    """The rank's share of a store: a contiguous range of units of
    ``unit_tokens`` tokens (whole requests), same cache and scales."""
    n_units = wl.num_tokens // unit_tokens
    lo, hi = shard_range(n_units, rank, world)
    t0, t1 = lo * unit_tokens, hi * unit_tokens
    return StoreWorkload(
        name=f"{wl.name}[{rank}/{world}]", num_tokens=t1 - t0,
        num_heads=wl.num_heads, head_size=wl.head_size,
        block_size=wl.block_size, num_blocks=wl.num_blocks, src=wl.src,
        key_offset=wl.key_offset + t0 * wl.key_stride0,
        key_stride0=wl.key_stride0,
        value_offset=wl.value_offset + t0 * wl.value_stride0,
        value_stride0=wl.value_stride0,
        slot_mapping=wl.slot_mapping[t0:t1].copy(), k_scale=wl.k_scale,
        v_scale=wl.v_scale, layout=wl.layout, flags=wl.flags,
        page_stride=wl.page_stride, dtype=wl.dtype)


def shard_gather(wl: GatherWorkload, rank: int, world: int):
    """The rank's share of a gather: a contiguous range of sequences, with
    cu_seq_lens rebased to 0.  Returns (sub-workload, first output row)."""
    lo, hi = shard_range(wl.num_seqs, rank, world)
    cu = wl.cu_seq_lens[lo: hi + 1].astype(np.int64)
    first = int(cu[0])
    sub = GatherWorkload(
        name=f"{wl.name}[{rank}/{world}]", block_size=wl.block_size,
        head_dim=wl.head_dim, num_blocks=wl.num_blocks, cache=wl.cache,
        block_table=wl.block_table[lo:hi].copy(),
        cu_seq_lens=(cu - first).astype(np.int32),
        block_stride=wl.block_stride)
    return sub, first


def sequences_of_store(wl: StoreWorkload, request_len: int):
    """Block table and cu_seq_lens that name the requests a "runs" store
    wrote (request r = tokens [r*request_len, (r+1)*request_len)), for
    reading them back: returns (block_table int32 [n, blocks per request],
    cu_seq_lens int32 [n + 1])."""
    B = wl.block_size
    n = wl.num_tokens // request_len
    bpr = (request_len + B - 1) // B
    first = wl.slot_mapping[: n * request_len].reshape(n, request_len)
    bt = (first[:, ::B][:, :bpr] // B).astype(np.int32)
    cu = (np.arange(n + 1, dtype=np.int64) * request_len).astype(np.int32)
    return bt, cu


def load_algorithmic_bytes(wl: StoreWorkload, block_table: np.ndarray,
                           cu_seq_lens: np.ndarray) -> int:
    """NVFP4 data + scale bytes read and bf16 rows written for every token
    the sequences name, plus the block-table entries and cu_seq_lens read."""
    H, D, B = wl.num_heads, wl.head_size, wl.block_size
    lens = np.diff(cu_seq_lens.astype(np.int64))
    n = int(lens.sum())
    entries = int(((lens + B - 1) // B).sum())
    return (n * 2 * H * (D // 2 + D // 16) + n * 2 * H * D * 2
            + 4 * entries + 4 * cu_seq_lens.size)


@dataclass
class IndexerStoreWorkload:
    """Inputs of one indexer-K store: K rows (bf16/fp16 bits, [T, D]) and
    their slots in a [num_blocks] cache of [B*D | B*4] blocks; the slots
    follow ``block_table`` / ``cu_seq_lens`` so a gather reads them back."""
    name: str
    k: np.ndarray
    num_tokens: int
    head_dim: int
    block_size: int
    num_blocks: int
    slot_mapping: np.ndarray
    block_table: np.ndarray
    cu_seq_lens: np.ndarray
    dtype: int = DTYPE_BF16

    @property
    def block_stride(self) -> int:
        return self.block_size * (self.head_dim + 4)

    def algorithmic_bytes(self) -> int:
        """K rows read, slots read, e4m3 rows and scales written."""
        n = int((self.slot_mapping >= 0).sum())
        return (self.num_tokens * (self.head_dim * 2 + 8)
                + n * (self.head_dim + 4))


def make_indexer_store(name: str, seed: int, seq_lens, block_size: int,
                       head_dim: int, num_blocks: int,
                       dtype: int = DTYPE_BF16,
                       spread: float = 2.0) -> IndexerStoreWorkload:
    """K rows N(0,1) times a per-token magnitude 10^U(-spread, spread), on
    the blocks of a random block table (sequences in cu order)."""
    rng = np.random.default_rng(seed)
    B, D = block_size, head_dim
    lens = np.asarray(seq_lens, dtype=np.int64)
    n = lens.size
    need = (lens + B - 1) // B
    mb = max(int(need.max()) if n else 1, 1)
    assert n * mb <= num_blocks
    bt = rng.permutation(num_blocks)[: n * mb].reshape(n, mb).astype(
        np.int32)
    cu = np.zeros(n + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    T = int(cu[-1])
    slots = np.concatenate(
        [bt[b, np.arange(m) // B].astype(np.int64) * B + np.arange(m) % B
         for b, m in enumerate(lens)] or [np.zeros(0, np.int64)])
    x = rng.standard_normal((T, D)).astype(np.float32)
    x *= (10.0 ** rng.uniform(-spread, spread, (T, 1))).astype(np.float32)
    if dtype == DTYPE_F16:
        x = np.clip(x, -60000, 60000)
    return IndexerStoreWorkload(
        name=name, k=element_bits(x.reshape(-1), dtype).reshape(T, D),
        num_tokens=T, head_dim=D, block_size=B, num_blocks=num_blocks,
        slot_mapping=slots.astype(np.int64), block_table=bt, cu_seq_lens=cu,
        dtype=dtype)


@dataclass
class AttentionWorkload:
    """Inputs of one paged decode-attention step over an NVFP4 cache: one
    query token per sequence (bf16/fp16 bits [n, Hq, D]), the cache pages
    (``num_blocks`` pages of ``page_stride`` bytes, K side at byte 0 of a
    page, V side at ``side_bytes``, HND unless ``layout``), the block table
    and the context lengths."""
    name: str
    query: np.ndarray
    num_kv_heads: int
    block_size: int
    num_blocks: int
    cache: np.ndarray
    block_table: np.ndarray
    context_lens: np.ndarray
    k_scale: np.float32
    v_scale: np.float32
    scale: np.float32
    layout: int = LAYOUT_HND
    flags: int = 0
    dtype: int = DTYPE_BF16

    @property
    def num_seqs(self) -> int:
        return self.query.shape[0]

    @property
    def num_q_heads(self) -> int:
        return self.query.shape[1]

    @property
    def head_size(self) -> int:
        return self.query.shape[2]

    @property
    def side_bytes(self) -> int:
        D = self.head_size
        return self.num_kv_heads * self.block_size * (D // 2 + D // 16)

    @property
    def page_stride(self) -> int:
        return 2 * self.side_bytes

    def algorithmic_bytes(self) -> int:
        """Every context token's NVFP4 K and V (data + scales) of every KV
        head read once, the queries read and the outputs written (2 bytes
        per element), block-table entries and context lengths read."""
        D, Hkv, B = self.head_size, self.num_kv_heads, self.block_size
        lens = self.context_lens.astype(np.int64)
        kv = int(lens.sum()) * Hkv * 2 * (D // 2 + D // 16)
        qo = 2 * self.query.size * 2
        meta = 4 * int(((lens + B - 1) // B).sum()) + 4 * lens.size
        return kv + qo + meta


def random_nvfp4_cache(rng, num_blocks: int, page_stride: int,
                       num_kv_heads: int, block_size: int, head_size: int,
                       sf_lo: int = 0x60, sf_hi: int = 0x7E) -> np.ndarray:
    """NVFP4 pages with uniform random data bytes (every e2m1 code) and
    scale bytes uniform over the e4m3 codes [sf_lo, sf_hi] (positive,
    never NaN) -- the range a per-tensor scale of amax/(448*6) gives
    N(0, 1) groups.  Bytes beyond 2*H*B*(D/2+S) per page are zero."""
    H, B, D = num_kv_heads, block_size, head_size
    data = H * B * D // 2
    side = data + H * B * D // 16
    cache = np.zeros((num_blocks, page_stride), dtype=np.uint8)
    for s in range(2):
        base = s * side
        cache[:, base:base + data] = rng.integers(
            0, 256, size=(num_blocks, data), dtype=np.uint8)
        cache[:, base + data:base + side] = rng.integers(
            sf_lo, sf_hi + 1, size=(num_blocks, side - data), dtype=np.uint8)
    return cache.reshape(-1)


def make_attention(name: str, seed: int, context_lens, num_q_heads: int,
                   num_kv_heads: int, head_size: int, block_size: int,
                   num_blocks: int = 0, dtype: int = DTYPE_BF16,
                   k_scale: float = 1.0 / 600.0, v_scale: float = 1.0 / 600.0,
                   scale: float | None = None, layout: int = LAYOUT_HND,
                   flags: int = 0, query_mult: float = 1.0,
                   extra_blocks: int = 0) -> AttentionWorkload:
    """Queries N(0, 1) x ``query_mult``; each sequence's pages are distinct
    random blocks of the cache (block table rows padded with further random
    blocks up to the longest sequence); cache bytes from
    ``random_nvfp4_cache``; softmax scale 1/sqrt(head_size) unless given."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(context_lens, dtype=np.int64)
    n, B = lens.size, block_size
    mb = max(int(((lens + B - 1) // B).max()) if n else 1, 1)
    nb = num_blocks or n * mb + extra_blocks
    assert n * mb <= nb
    bt = rng.permutation(nb)[: n * mb].reshape(n, mb).astype(np.int32)
    D = head_size
    page_stride = 2 * num_kv_heads * B * (D // 2 + D // 16)
    cache = random_nvfp4_cache(rng, nb, page_stride, num_kv_heads, B, D)
    q = rng.standard_normal((n, num_q_heads, D)).astype(np.float32)
    q *= np.float32(query_mult)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    return AttentionWorkload(
        name=name, query=element_bits(q.reshape(-1), dtype).reshape(q.shape),
        num_kv_heads=num_kv_heads, block_size=B, num_blocks=nb, cache=cache,
        block_table=bt, context_lens=lens.astype(np.int32),
        k_scale=np.float32(k_scale), v_scale=np.float32(v_scale),
        scale=np.float32(scale), layout=layout, flags=flags, dtype=dtype)


def attention_workload(seed: int = 5, num_seqs: int = 200) -> AttentionWorkload:
    """``llama70b_decode`` -- one decode step of Llama-3.1-70B-shaped
    attention (64 query heads, 8 KV heads, head_size 128) over an NVFP4
    cache with block_size 16: ``num_seqs`` sequences (the 200-prompt
    serving runs) whose contexts are a 512-token prompt plus U[0, 2048]
    generated tokens."""
    rng = np.random.default_rng(seed)
    lens = 512 + rng.integers(0, 2049, size=num_seqs)
    return make_attention("llama70b_decode", seed, lens, num_q_heads=64,
                          num_kv_heads=8, head_size=128, block_size=16)
