"""Seeded synthetic inputs for paged MLA decode.

This module is shared by the tests, the benchmark and the smoke check.  It
only draws random numbers and writes them into the storage formats; it holds
none of the attention arithmetic.  The FP8 cache rows are produced with
torch's own float8_e4m3fn cast (a library routine).

Storage formats (one KV head, page size 64):
  q            bf16  [batch, s_q, h_q, 576]
  kvcache bf16 bf16  [num_pages, page_size, 1, 576]
  kvcache fp8  uint8 [num_pages, page_size, 1, 656]: bytes [0,512) e4m3 codes
               of dims 0..511, [512,528) four little-endian float32 scales
               (scale k covers dims [128k, 128k+128)), [528,656) 64 bf16
               RoPE values (dims 512..575)
  block_table  int32 [batch, max_blocks]  (unused slots hold 0)
  cache_seqlens int32 [batch]
  indices      int32 [batch, s_q, topk] logical token ids, -1 = unused

The five named workloads follow the decode shapes of the FlashMLA article
("Why FlashMLA's decode kernel reaches 660 TFLOPS": h_q = 128 with s_q = 2
for the compute-bound case, top-k 2048 / 32768 for sparse FP8 decode) plus a
tiny case and a small-head memory-bound case.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional, Tuple

import numpy as np
import torch

D_QK = 576
D_V = 512
D_ROPE = 64
FP8_ROW_BYTES = 656
PAGE_SIZE = 64
E4M3_MAX = 448.0


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    h_q: int
    s_q: int
    mode: str                                   # "dense" (bf16 cache) or "sparse" (fp8 cache + indices)
    seqlens: Optional[Tuple[int, ...]] = None   # explicit lengths
    seqlen_range: Optional[Tuple[int, int]] = None  # uniform integer [lo, hi]
    seqlen: Optional[int] = None                # fixed length
    topk: int = 0
    causal: bool = False
    invalid_frac: float = 0.05                  # sparse: trailing fraction of each index row set to -1
    page_size: int = PAGE_SIZE
    sm_scale: Optional[float] = None            # default 1/sqrt(576)
    fp8: Optional[bool] = None                  # cache format; None: FP8 for sparse, bf16 for dense
    fp8_scales: str = "tile"                    # FP8 rows: "tile" = 656 B, four scales in the row;
                                                # "token" = 640 B rows + one fp32 scale per token
    ragged_topk: bool = False                   # sparse: per-row topk_lengths; slots past them hold ids

    @property
    def is_fp8(self) -> bool:
        return self.fp8 if self.fp8 is not None else self.mode == "sparse"

    @property
    def scale(self) -> float:
        return self.sm_scale if self.sm_scale is not None else 1.0 / math.sqrt(D_QK)


WORKLOADS = {
    "tiny": Workload("tiny", batch=2, h_q=16, s_q=1, mode="dense", seqlens=(100, 257)),
    "dense_membound": Workload("dense_membound", batch=128, h_q=16, s_q=1, mode="dense",
                               seqlen_range=(1024, 8192)),
    "dense_computebound": Workload("dense_computebound", batch=64, h_q=128, s_q=2, mode="dense",
                                   seqlen=4096, causal=True),
    "sparse_fp8": Workload("sparse_fp8", batch=128, h_q=128, s_q=2, mode="sparse", seqlen=32768,
                           topk=2048),
    "sparse_fp8_long": Workload("sparse_fp8_long", batch=16, h_q=128, s_q=1, mode="sparse",
                                seqlen_range=(65536, 131072), topk=32768),
    # mode variant: the memory-bound dense mix over the FP8 cache (656 bytes per token)
    "dense_membound_fp8": Workload("dense_membound_fp8", batch=128, h_q=16, s_q=1, mode="dense",
                                   seqlen_range=(1024, 8192), fp8=True),
    # mode variant: the sparse FP8 shape over the bf16 cache (1152 bytes per gathered row)
    "sparse_bf16": Workload("sparse_bf16", batch=128, h_q=128, s_q=2, mode="sparse", seqlen=32768, topk=2048,
                            fp8=False),
    # mode variant: the sparse FP8 shape over 640-byte rows with one scale per token
    "sparse_fp8_token": Workload("sparse_fp8_token", batch=128, h_q=128, s_q=2, mode="sparse", seqlen=32768,
                                 topk=2048, fp8_scales="token"),
}
# Seed per named workload: 1000 + its position (1-based) in the list above.
SEEDS = {name: 1000 + i for i, name in enumerate(WORKLOADS, start=1)}


@dataclass(frozen=True)
class PrefillWorkload:
    """Sparse prefill: s_q query tokens, each attending to topk rows of one
    unpaged bf16 KV of s_kv rows (no batch dimension)."""
    name: str
    s_q: int
    s_kv: int
    h_q: int
    topk: int
    invalid_frac: float = 0.0                   # trailing fraction of each index row set to -1
    sm_scale: Optional[float] = None            # default 1/sqrt(576)

    @property
    def scale(self) -> float:
        return self.sm_scale if self.sm_scale is not None else 1.0 / math.sqrt(D_QK)


# The prefill shape the FlashMLA article's sparse-prefill kernel is quoted on
# is not printed; 128 heads and top-k 2048 follow its sparse decode numbers,
# a 4096-token prefill chunk attends into a 32768-row KV.
PREFILL_WORKLOADS = {
    "prefill_tiny": PrefillWorkload("prefill_tiny", s_q=5, s_kv=300, h_q=16, topk=100, invalid_frac=0.1),
    "sparse_prefill": PrefillWorkload("sparse_prefill", s_q=4096, s_kv=32768, h_q=128, topk=2048),
}
PREFILL_SEEDS = {name: 1100 + i for i, name in enumerate(PREFILL_WORKLOADS, start=1)}


@dataclass
class PrefillInputs:
    workload: PrefillWorkload
    q: torch.Tensor        # bf16 [s_q, h_q, 576]
    kv: torch.Tensor       # bf16 [s_kv, 576]
    indices: torch.Tensor  # int32 [s_q, topk]
    sm_scale: float
    seed: int

    def to(self, device) -> "PrefillInputs":
        return PrefillInputs(self.workload, self.q.to(device), self.kv.to(device), self.indices.to(device),
                             self.sm_scale, self.seed)


def make_prefill_inputs(w, seed: Optional[int] = None, device="cpu") -> PrefillInputs:
    """q and kv ~ N(0, 1) in bf16 (torch generator on ``device``); each query
    token's index row holds distinct ids drawn uniformly from [0, s_kv) (numpy
    PCG64), its trailing ``invalid_frac`` part set to -1."""
    if isinstance(w, str):
        if seed is None:
            seed = PREFILL_SEEDS[w]
        w = PREFILL_WORKLOADS[w]
    if seed is None:
        seed = 4321
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = torch.randn((w.s_q, w.h_q, D_QK), generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    kv = torch.randn((w.s_kv, D_QK), generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    idx = np.full((w.s_q, w.topk), -1, dtype=np.int32)
    n_valid = min(w.topk - int(math.floor(w.invalid_frac * w.topk)), w.s_kv)
    for i in range(w.s_q):
        if n_valid > 0:
            idx[i, :n_valid] = rng.choice(w.s_kv, size=n_valid, replace=False).astype(np.int32)
    return PrefillInputs(w, q, kv, torch.from_numpy(idx).to(device), w.scale, seed)


@dataclass
class Inputs:
    workload: Workload
    q: torch.Tensor
    kvcache: torch.Tensor
    block_table: torch.Tensor
    cache_seqlens: torch.Tensor
    indices: Optional[torch.Tensor]
    sm_scale: float
    seed: int
    meta: dict = field(default_factory=dict)
    kv_scales: Optional[torch.Tensor] = None      # fp32 [num_pages, page_size] ("token" FP8 rows)
    topk_lengths: Optional[torch.Tensor] = None   # int32 [batch, s_q] (ragged top-k)

    def to(self, device) -> "Inputs":
        mv = lambda t: None if t is None else t.to(device)
        return Inputs(self.workload, mv(self.q), mv(self.kvcache), mv(self.block_table),
                      mv(self.cache_seqlens), mv(self.indices), self.sm_scale, self.seed,
                      dict(self.meta), mv(self.kv_scales), mv(self.topk_lengths))


def describe_lengths(w: Workload) -> str:
    """The length rule of a workload, in words (for reports)."""
    seed = SEEDS.get(w.name)
    if w.seqlens is not None:
        return f"fixed {list(w.seqlens)}"
    if w.seqlen is not None:
        return f"all {w.seqlen}"
    return f"uniform int [{w.seqlen_range[0]}, {w.seqlen_range[1]}], seed {seed}"


def draw_seqlens(w: Workload, rng: np.random.Generator) -> np.ndarray:
    if w.seqlens is not None:
        lens = np.asarray(w.seqlens, dtype=np.int64)
        assert lens.shape == (w.batch,)
        return lens
    if w.seqlen is not None:
        return np.full((w.batch,), w.seqlen, dtype=np.int64)
    lo, hi = w.seqlen_range
    return rng.integers(lo, hi + 1, size=w.batch, dtype=np.int64)


def _paging(lens: np.ndarray, page_size: int, rng: np.random.Generator):
    """Random permutation of exactly sum(ceil(len/page)) pages shared by all elements."""
    nblk = (lens + page_size - 1) // page_size
    total = int(nblk.sum())
    perm = rng.permutation(total).astype(np.int32)
    width = max(1, int(nblk.max()) if len(nblk) else 1)
    table = np.zeros((len(lens), width), dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[off:off + n]
        off += n
    return table, max(total, 1)


def _normal_bf16(n_rows: int, gen: torch.Generator, device) -> torch.Tensor:
    return torch.randn((n_rows, D_QK), generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def encode_fp8_rows(x: torch.Tensor) -> torch.Tensor:
    """Source values [n, 576] float32 -> [n, 656] uint8 rows in the FP8 cache format.

    Each 1x128 tile of dims 0..511 gets scale = amax/448 (float32; scale 1 for
    an all-zero tile) and codes = float8_e4m3fn(x / scale) via torch's cast;
    dims 512..575 are stored as bf16.
    """
    n = x.shape[0]
    nope = x[:, :D_V].float().reshape(n, 4, 128)
    amax = nope.abs().amax(dim=2)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    codes = (nope / scale[:, :, None]).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    rope = x[:, D_V:].to(torch.bfloat16)
    row = torch.empty((n, FP8_ROW_BYTES), dtype=torch.uint8, device=x.device)
    row[:, :D_V] = codes.reshape(n, D_V).view(torch.uint8)
    row[:, D_V:D_V + 16] = scale.contiguous().view(torch.uint8).reshape(n, 16)
    row[:, D_V + 16:] = rope.contiguous().view(torch.uint8).reshape(n, 2 * D_ROPE)
    return row


def encode_fp8_token_rows(x: torch.Tensor):
    """Source values [n, 576] float32 -> ([n, 640] uint8 rows, [n] fp32 scales): one scale per
    token, amax of dims 0..511 / 448 (1 for an all-zero token), codes = float8_e4m3fn(x / scale)
    via torch's cast in bytes [0, 512), dims 512..575 as bf16 in bytes [512, 640)."""
    n = x.shape[0]
    nope = x[:, :D_V].float()
    amax = nope.abs().amax(dim=1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    codes = (nope / scale[:, None]).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    row = torch.empty((n, 640), dtype=torch.uint8, device=x.device)
    row[:, :D_V] = codes.view(torch.uint8)
    row[:, D_V:] = x[:, D_V:].to(torch.bfloat16).contiguous().view(torch.uint8).reshape(n, 2 * D_ROPE)
    return row, scale.contiguous()


def make_inputs(w, seed: Optional[int] = None, device="cpu", poison_tail: bool = True,
                chunk_pages: int = 2048) -> Inputs:
    """Draw one batch of inputs for workload ``w`` (a Workload or a name in WORKLOADS).

    Structure (lengths, page permutation, indices) comes from numpy's PCG64
    seeded with ``seed``; values (q, kv) from a torch generator with the same
    seed on ``device``.  With ``poison_tail`` the unused slots of each
    element's last page hold NaN so that any read past the length shows.
    """
    if isinstance(w, str):
        if seed is None:
            seed = SEEDS[w]
        w = WORKLOADS[w]
    if seed is None:
        seed = 1234
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    lens = draw_seqlens(w, rng)
    table, num_pages = _paging(lens, w.page_size, rng)

    q = torch.randn((w.batch, w.s_q, w.h_q, D_QK), generator=gen, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    ntok = num_pages * w.page_size
    per_token = w.is_fp8 and w.fp8_scales == "token"
    row_bytes = 640 if per_token else FP8_ROW_BYTES
    kv_scales = torch.empty((ntok,), dtype=torch.float32, device=device) if per_token else None
    if w.is_fp8:
        kv = torch.empty((ntok, row_bytes), dtype=torch.uint8, device=device)
    else:
        kv = torch.empty((ntok, D_QK), dtype=torch.bfloat16, device=device)
    step = chunk_pages * w.page_size
    for t0 in range(0, ntok, step):
        t1 = min(ntok, t0 + step)
        x = torch.randn((t1 - t0, D_QK), generator=gen, device=device, dtype=torch.float32)
        if per_token:
            kv[t0:t1], kv_scales[t0:t1] = encode_fp8_token_rows(x)
        else:
            kv[t0:t1] = encode_fp8_rows(x) if w.is_fp8 else x.to(torch.bfloat16)

    if poison_tail:
        for b, L in enumerate(lens.tolist()):
            nblk = (L + w.page_size - 1) // w.page_size
            used = L - (nblk - 1) * w.page_size if nblk else 0
            if nblk == 0 or used == w.page_size:
                continue
            page = int(table[b, nblk - 1])
            s0 = page * w.page_size + used
            s1 = (page + 1) * w.page_size
            if w.is_fp8:
                kv[s0:s1] = 0x7F  # e4m3 NaN codes; scale / RoPE bytes 0x7F7F.. are NaN too
                if per_token:
                    kv_scales[s0:s1] = float("nan")
            else:
                kv[s0:s1] = float("nan")

    indices = None
    if w.mode == "sparse":
        indices_np = np.full((w.batch, w.s_q, w.topk), -1, dtype=np.int32)
        n_invalid = int(math.floor(w.invalid_frac * w.topk))
        n_valid = w.topk - n_invalid
        for b in range(w.batch):
            L = int(lens[b])
            for i in range(w.s_q):
                k = min(n_valid, L)
                if k > 0:
                    indices_np[b, i, :k] = rng.choice(L, size=k, replace=False).astype(np.int32)
        indices = torch.from_numpy(indices_np).to(device)

    topk_lengths = None
    if w.mode == "sparse" and w.ragged_topk:
        # per row a length uniform in [0, topk]; the slots past it hold ids that
        # would be valid (they must be ignored, not merely skipped as -1)
        tl = rng.integers(0, w.topk + 1, size=(w.batch, w.s_q)).astype(np.int32)
        idx_np = indices.cpu().numpy()
        for b in range(w.batch):
            L = int(lens[b])
            for i in range(w.s_q):
                if L > 0:
                    idx_np[b, i, tl[b, i]:] = rng.integers(0, L, size=w.topk - tl[b, i])
        indices = torch.from_numpy(idx_np).to(device)
        topk_lengths = torch.from_numpy(tl).to(device)

    kv = kv.reshape(num_pages, w.page_size, 1, (row_bytes if w.is_fp8 else D_QK))
    return Inputs(w, q, kv, torch.from_numpy(table).to(device),
                  torch.from_numpy(lens.astype(np.int32)).to(device), indices, w.scale, seed,
                  meta={"num_pages": num_pages},
                  kv_scales=None if kv_scales is None else kv_scales.reshape(num_pages, w.page_size),
                  topk_lengths=topk_lengths)


def custom(name="custom", **kw) -> Workload:
    """A Workload with explicit fields (tests)."""
    return Workload(name=name, **kw)


def with_fields(w: Workload, **kw) -> Workload:
    return replace(w, **kw)



# ----------------------------------------------------------------------------
# FP8 top-k indexer inputs
# ----------------------------------------------------------------------------
IDX_DIM = 128


@dataclass(frozen=True)
class IndexWorkload:
    """Index queries of n_new tokens per element (ragged rows, the last n_new
    positions of each element's cache) scored against a paged FP8 key cache."""
    name: str
    batch: int
    n_new: int                                  # query tokens per element
    h_idx: int                                  # index heads
    topk: int
    seqlens: Optional[Tuple[int, ...]] = None
    seqlen: Optional[int] = None
    seqlen_range: Optional[Tuple[int, int]] = None
    relu: bool = False
    rows: Optional[Tuple[int, ...]] = None      # ragged: query tokens per element (overrides n_new)


# 64 index heads of dimension 128 and top-k 2048 are the shapes the sparse
# decode workloads consume (the pages give the indexer no shapes).
INDEX_WORKLOADS = {
    "index_tiny": IndexWorkload("index_tiny", batch=2, n_new=2, h_idx=8, topk=64, seqlens=(300, 90)),
    "index_decode": IndexWorkload("index_decode", batch=128, n_new=2, h_idx=64, topk=2048, seqlen=32768),
}
INDEX_SEEDS = {name: 1200 + i for i, name in enumerate(INDEX_WORKLOADS, start=1)}


@dataclass
class IndexInputs:
    workload: IndexWorkload
    q_codes: torch.Tensor       # uint8 [num_tokens, h_idx, 128] E4M3 codes
    q_scales: torch.Tensor      # fp32 [num_tokens, h_idx]
    weights: torch.Tensor       # fp32 [num_tokens, h_idx]
    row_offsets: torch.Tensor   # int32 [batch + 1]
    k_codes: torch.Tensor       # uint8 [num_pages, 64, 128]
    k_scales: torch.Tensor      # fp32 [num_pages, 64]
    block_table: torch.Tensor   # int32 [batch, max_blocks]
    cache_seqlens: torch.Tensor  # int32 [batch]
    topk: int
    relu: bool
    seed: int

    def to(self, device) -> "IndexInputs":
        f = lambda t: t.to(device)
        return IndexInputs(self.workload, f(self.q_codes), f(self.q_scales), f(self.weights), f(self.row_offsets),
                           f(self.k_codes), f(self.k_scales), f(self.block_table), f(self.cache_seqlens),
                           self.topk, self.relu, self.seed)


def quantize_e4m3_rows(x: torch.Tensor):
    """[..., 128] float32 -> (E4M3 codes uint8 [..., 128], fp32 scales [...]): scale = amax / 448
    (1 for an all-zero row), codes = torch's float8_e4m3fn cast of x / scale."""
    amax = x.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    codes = (x / scale[..., None]).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def make_index_inputs(w, seed: Optional[int] = None, device="cpu") -> IndexInputs:
    """Keys and queries ~ N(0, 1) quantised per 128-dim row; weights ~ N(0, 1) / sqrt(h_idx);
    lengths and a random page permutation as for decode (numpy PCG64 with ``seed``)."""
    if isinstance(w, str):
        if seed is None:
            seed = INDEX_SEEDS[w]
        w = INDEX_WORKLOADS[w]
    if seed is None:
        seed = 2468
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dw = Workload(w.name, batch=w.batch, h_q=1, s_q=1, mode="dense", seqlens=w.seqlens, seqlen=w.seqlen,
                  seqlen_range=w.seqlen_range)
    lens = draw_seqlens(dw, rng)
    assert np.all(lens >= 0)
    table, num_pages = _paging(lens, PAGE_SIZE, rng)
    counts = np.asarray(w.rows if w.rows is not None else [w.n_new] * w.batch, dtype=np.int64)
    assert counts.shape == (w.batch,)
    n = int(counts.sum())
    qx = torch.randn((n, w.h_idx, IDX_DIM), generator=gen, device=device, dtype=torch.float32)
    q_codes, q_scales = quantize_e4m3_rows(qx)
    weights = torch.randn((n, w.h_idx), generator=gen, device=device, dtype=torch.float32) / math.sqrt(w.h_idx)
    kx = torch.randn((num_pages * PAGE_SIZE, IDX_DIM), generator=gen, device=device, dtype=torch.float32)
    k_codes, k_scales = quantize_e4m3_rows(kx)
    offs = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32))
    return IndexInputs(w, q_codes.contiguous(), q_scales.contiguous(), weights.contiguous(), offs.to(device),
                       k_codes.reshape(num_pages, PAGE_SIZE, IDX_DIM).contiguous(),
                       k_scales.reshape(num_pages, PAGE_SIZE).contiguous(), torch.from_numpy(table).to(device),
                       torch.from_numpy(lens.astype(np.int32)).to(device), w.topk, w.relu, seed)
