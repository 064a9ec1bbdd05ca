"""Seeded synthetic workloads for the paged two-family prep + attention path.

This module only draws inputs: raw bf16 activations, norm weights, request
lengths and page tables. It computes none of the method's arithmetic (no norm,
no rotary table, no slot addressing, no attention); both the CUDA path and the
fp64 oracle consume what it returns.

Shapes follow the serving geometry of the "paged KV serving across both
attention families" page (Description): local layers are head_dim 256 with 8
KV heads under a sliding window, global layers are head_dim 512 with 1 KV
head under full causal attention, 16 query heads, page size 16.

Random numbers: numpy ``PCG64(seed)``, seed = 1000 + config index unless given.
bf16 values are float32 draws rounded to bfloat16 (round to nearest even) and
returned as raw ``uint16`` bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

PAGE_SIZE = 16
EPS = 1e-6
SM_SCALE = 1.0
POOL_SENTINEL = 0xFFFF  # a bf16 NaN bit pattern; never produced by the kernels


@dataclass(frozen=True)
class Family:
    """One attention family's head geometry and per-call policy."""

    name: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    rope_theta: float
    window_left: int


HD256 = Family("hd256", 16, 8, 256, 1.0e4, 1023)
HD512 = Family("hd512", 16, 1, 512, 1.0e6, -1)


@dataclass
class Batch:
    """Ragged request batch in the page-table form the plan consumes."""

    qo_indptr: np.ndarray        # int64 [R+1]
    kv_page_indptr: np.ndarray   # int64 [R+1]
    page_ids: np.ndarray         # int32 [sum pages]
    last_page_len: np.ndarray    # int32 [R]
    start_pos: np.ndarray        # int64 [R]
    page_size: int
    num_pages: int               # pages in the pool the ids index

    @property
    def num_req(self) -> int:
        return len(self.start_pos)

    @property
    def num_tokens(self) -> int:
        return int(self.qo_indptr[-1])

    @property
    def qo_lens(self) -> np.ndarray:
        return np.diff(self.qo_indptr)


@dataclass
class FamilyInputs:
    """Everything one family's prep + attention call consumes."""

    family: Family
    batch: Batch
    num_layers: int
    layer: int
    q_raw: np.ndarray            # uint16 bf16 bits [T, Hq, D]
    k_raw: np.ndarray            # uint16 bf16 bits [T, Hkv, D]
    v_raw: np.ndarray | None     # uint16 bf16 bits [T, Hkv, D] (hd256 only)
    w_q: np.ndarray              # uint16 bf16 bits [D]
    w_k: np.ndarray              # uint16 bf16 bits [D]
    pool_fill: str               # "sentinel" or "normal"
    pool_seed: int
    eps: float = EPS
    sm_scale: float = SM_SCALE

    @property
    def pool_shape(self) -> tuple:
        f, b = self.family, self.batch
        return (self.num_layers, b.num_pages, 2, f.num_kv_heads, b.page_size, f.head_dim)

    @property
    def rope_rows(self) -> int:
        b = self.batch
        return int(np.max(b.start_pos + b.qo_lens)) if b.num_req else 1

    def make_pool(self) -> np.ndarray:
        """The pool's initial contents as bf16 bits, [L, P, 2, Hkv, ps, D]."""
        if self.pool_fill == "sentinel":
            return np.full(self.pool_shape, POOL_SENTINEL, dtype=np.uint16)
        rng = np.random.Generator(np.random.PCG64(self.pool_seed))
        return bf16_normal(rng, self.pool_shape)


@dataclass
class Workload:
    name: str
    description: str
    families: list = field(default_factory=list)   # list[FamilyInputs]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); finite inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_normal(rng: np.random.Generator, shape, mean: float = 0.0, std: float = 1.0,
                chunk: int = 1 << 24) -> np.ndarray:
    """bf16 bit patterns of N(mean, std^2) float32 draws, generated in chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        if mean != 0.0:
            x += np.float32(mean)
        out[s:e] = f32_to_bf16_bits(x)
    return out.reshape(shape)


def make_batch(rng: np.random.Generator, qo_lens, start_pos, page_size: int,
               num_pages: int | None = None, spare_pages: int = 0) -> Batch:
    """Page table for requests holding KV positions [0, start_pos + qo_len).

    Each request holds ceil(kv_len / page_size) pages; the ids are the leading
    entries of a seeded permutation of the whole pool, so pages are scattered.
    """
    qo_lens = np.asarray(qo_lens, dtype=np.int64)
    start_pos = np.asarray(start_pos, dtype=np.int64)
    kv_lens = start_pos + qo_lens
    npages = (kv_lens + page_size - 1) // page_size
    need = int(npages.sum())
    if num_pages is None:
        num_pages = need + spare_pages
    if need > num_pages:
        raise ValueError(f"pool of {num_pages} pages cannot hold {need}")
    perm = rng.permutation(num_pages).astype(np.int32)
    qo_indptr = np.zeros(len(qo_lens) + 1, np.int64)
    qo_indptr[1:] = np.cumsum(qo_lens)
    kv_page_indptr = np.zeros(len(qo_lens) + 1, np.int64)
    kv_page_indptr[1:] = np.cumsum(npages)
    last = (kv_lens - (npages - 1) * page_size).astype(np.int32)
    return Batch(qo_indptr, kv_page_indptr, perm[:need].copy(), last, start_pos,
                 page_size, int(num_pages))


def family_inputs(rng: np.random.Generator, fam: Family, batch: Batch, num_layers: int,
                  layer: int, pool_fill: str, pool_seed: int) -> FamilyInputs:
    T = batch.num_tokens
    q = bf16_normal(rng, (T, fam.num_qo_heads, fam.head_dim))
    k = bf16_normal(rng, (T, fam.num_kv_heads, fam.head_dim))
    v = bf16_normal(rng, (T, fam.num_kv_heads, fam.head_dim)) if fam.head_dim == 256 else None
    w_q = bf16_normal(rng, (fam.head_dim,), mean=1.0, std=0.1)
    w_k = bf16_normal(rng, (fam.head_dim,), mean=1.0, std=0.1)
    return FamilyInputs(fam, batch, num_layers, layer, q, k, v, w_q, w_k, pool_fill, pool_seed)


def _with_window(fam: Family, w: int) -> Family:
    return Family(fam.name, fam.num_qo_heads, fam.num_kv_heads, fam.head_dim, fam.rope_theta, w)


CONFIG_NAMES = {
    1: "hd256 prefill, 1 request x 9 tokens, window_left 3, 4-page pool",
    2: "hd512 prefill, 1 request x 512 tokens, full causal, 64-page pool",
    3: "hd256 batched ragged prefill, 8 requests x U[128,2048] tokens, window_left 1023, "
       "4 layers x 8192 pages (layer 2)",
    4: "dual-family decode step, 64 requests x 1 token, existing KV U[1,1024] (hd256, "
       "window_left 1023) and U[1,16384] (hd512, full causal)",
    5: "long prefill, 1 request x 16384 tokens, hd256 window_left 1023 + hd512 full causal",
}


def make_workload(index: int, seed: int | None = None, pool_fill: str | None = None) -> Workload:
    """Build config ``index`` (1..5). ``pool_fill`` overrides the pool's initial fill."""
    seed = 1000 + index if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    wl = Workload(f"cfg{index}", CONFIG_NAMES[index])
    ps = PAGE_SIZE
    if index == 1:
        b = make_batch(rng, [9], [0], ps, num_pages=4)
        wl.families.append(family_inputs(rng, _with_window(HD256, 3), b, 1, 0,
                                         pool_fill or "sentinel", seed + 1))
    elif index == 2:
        b = make_batch(rng, [512], [0], ps, num_pages=64)
        wl.families.append(family_inputs(rng, HD512, b, 1, 0, pool_fill or "sentinel", seed + 1))
    elif index == 3:
        lens = rng.integers(128, 2048, size=8, endpoint=True)
        b = make_batch(rng, lens, np.zeros(8, np.int64), ps, num_pages=8192)
        wl.families.append(family_inputs(rng, HD256, b, 4, 2, pool_fill or "sentinel", seed + 1))
    elif index == 4:
        R = 64
        l256 = rng.integers(1, 1024, size=R, endpoint=True)
        l512 = rng.integers(1, 16384, size=R, endpoint=True)
        b256 = make_batch(rng, np.ones(R, np.int64), l256, ps, spare_pages=64)
        b512 = make_batch(rng, np.ones(R, np.int64), l512, ps, spare_pages=64)
        wl.families.append(family_inputs(rng, HD256, b256, 1, 0, pool_fill or "normal", seed + 1))
        wl.families.append(family_inputs(rng, HD512, b512, 1, 0, pool_fill or "normal", seed + 2))
    elif index == 5:
        T = 16384
        b256 = make_batch(rng, [T], [0], ps, num_pages=1024)
        b512 = make_batch(rng, [T], [0], ps, num_pages=1024)
        wl.families.append(family_inputs(rng, HD256, b256, 1, 0, pool_fill or "sentinel", seed + 1))
        wl.families.append(family_inputs(rng, HD512, b512, 1, 0, pool_fill or "sentinel", seed + 2))
    else:
        raise ValueError(f"no config {index}")
    return wl


def custom_family(fam: Family, qo_lens, start_pos, seed: int, num_pages: int | None = None,
                  num_layers: int = 1, layer: int = 0, page_size: int = PAGE_SIZE,
                  spare_pages: int = 8, pool_fill: str = "sentinel",
                  window_left: int | None = None) -> FamilyInputs:
    """A seeded single-family case with explicit lengths (tests and edge cases)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    b = make_batch(rng, qo_lens, start_pos, page_size, num_pages=num_pages,
                   spare_pages=spare_pages)
    if window_left is not None:
        fam = _with_window(fam, window_left)
    return family_inputs(rng, fam, b, num_layers, layer, pool_fill, seed + 1)


@dataclass
class CascadeInputs:
    """Requests sharing a key prefix, in three page tables over one pool.

    ``full`` holds each request's keys [0, L_r) in its own pages; ``prefix`` lists the
    shared prefix pages (keys [0, prefix_len)) for every request; ``suffix`` holds each
    request's keys [prefix_len, L_r) from slot 0 of its own pages. ``hist_k`` / ``hist_v``
    are every request's key and value rows by position (bf16 bits [L_r, Hkv, D]; the prefix
    rows are the same for every request). Filling the pool from them is left to the caller.
    The queries are each request's last ``step_lens[r]`` positions.
    """

    q: np.ndarray                # uint16 bf16 bits [T, Hq, D]
    hist_k: list
    hist_v: list
    full: Batch
    prefix: Batch
    suffix: Batch
    prefix_len: int
    num_kv_heads: int
    head_dim: int


def make_cascade(rng: np.random.Generator, prefix_len: int, suffix_lens, step_lens,
                 page_size: int, num_qo_heads: int, num_kv_heads: int,
                 head_dim: int) -> CascadeInputs:
    suffix_lens = np.asarray(suffix_lens, np.int64)
    step_lens = np.asarray(step_lens, np.int64)
    if (step_lens > suffix_lens).any() or (step_lens < 1).any():
        raise ValueError("each step must lie inside its request's own suffix")
    R = len(suffix_lens)
    L = prefix_len + suffix_lens
    pre_k = bf16_normal(rng, (prefix_len, num_kv_heads, head_dim))
    pre_v = bf16_normal(rng, (prefix_len, num_kv_heads, head_dim))
    hist_k, hist_v = [], []
    for r in range(R):
        hist_k.append(np.concatenate([pre_k, bf16_normal(rng, (int(suffix_lens[r]), num_kv_heads, head_dim))]))
        hist_v.append(np.concatenate([pre_v, bf16_normal(rng, (int(suffix_lens[r]), num_kv_heads, head_dim))]))
    ceil = lambda n: -(-np.asarray(n, np.int64) // page_size)
    n_pre = int(ceil(prefix_len))
    n_suf = ceil(suffix_lens)
    n_full = ceil(L)
    total = n_pre + int(n_suf.sum()) + int(n_full.sum())
    perm = rng.permutation(total).astype(np.int32)
    pre_pages, off = perm[:n_pre], n_pre
    suf_pages, full_pages = [], []
    for r in range(R):
        suf_pages.append(perm[off:off + n_suf[r]])
        off += int(n_suf[r])
    for r in range(R):
        full_pages.append(perm[off:off + n_full[r]])
        off += int(n_full[r])
    qo = np.zeros(R + 1, np.int64)
    qo[1:] = np.cumsum(step_lens)
    start = (L - step_lens).astype(np.int64)

    def table(pages, lens):
        indptr = np.zeros(R + 1, np.int64)
        indptr[1:] = np.cumsum([len(p) for p in pages])
        lens = np.asarray(lens, np.int64)
        last = (lens - (ceil(lens) - 1) * page_size).astype(np.int32)
        return Batch(qo.copy(), indptr, np.concatenate(pages).astype(np.int32), last,
                     start.copy(), page_size, total)

    q = bf16_normal(rng, (int(qo[-1]), num_qo_heads, head_dim))
    return CascadeInputs(q, hist_k, hist_v, table(full_pages, L),
                         table([pre_pages] * R, [prefix_len] * R), table(suf_pages, suffix_lens),
                         prefix_len, num_kv_heads, head_dim)
