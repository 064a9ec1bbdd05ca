"""ctypes binding of ``libpg.so`` (declared in ``include/pg.h``).

Argument marshalling only: every step of the path runs in the library's
kernels. Device buffers are passed as torch CUDA tensors (their ``data_ptr``),
host plan inputs as numpy arrays, streams as ``torch.cuda.Stream`` (default:
torch's current stream). Each ``pg_*`` function returns the library's status
code; ``check`` turns a nonzero code into ``PgError``.

Importing this module loads the library and raises ``ImportError`` if it has not
been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpg.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python -c 'import __graft_entry__ as g; g.build()'`")
_lib = C.CDLL(LIB_PATH)

# status codes (include/pg.h)
PG_OK = 0
PG_ERR_ARG = -1
PG_ERR_PAGE_OOB = -2
PG_ERR_LAST_PAGE_LEN = -3
PG_ERR_I32_OVERFLOW = -4
PG_ERR_ZERO_KV_HEADS = -5
PG_ERR_HEADS = -6
PG_ERR_NONFINITE = -7
PG_ERR_ROPE_RANGE = -8
PG_ERR_COVERAGE = -9
PG_ERR_LAYER = -10
PG_ERR_LAYOUT = -11
PG_ERR_PLAN_MISMATCH = -12
PG_ERR_WINDOW = -13
PG_ERR_WORKSPACE = -14
PG_ERR_STREAM = -15
PG_ERR_CUDA = -16
PG_ERR_DEVICE_BOUNDS = -17
PG_ERR_ALIGN = -18
PG_ERR_DEVICE_TIMEOUT = -19


class PgError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {pg_status_string(status)} ({status})")


class pg_pool_t(C.Structure):
    _fields_ = [("base", C.c_void_p),
                ("num_layers", C.c_int32), ("num_pages", C.c_int32), ("page_size", C.c_int32),
                ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("stride_layer", C.c_int64), ("stride_page", C.c_int64), ("stride_kv", C.c_int64),
                ("stride_head", C.c_int64), ("stride_slot", C.c_int64),
                ("capacity", C.c_int64)]


class pg_plan_info_t(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "num_req", "num_tokens", "num_qo_heads", "num_kv_heads", "head_dim", "page_size",
        "max_page_id", "max_last_page_len", "max_qo_len", "max_kv_len", "max_pos_end",
        "cta_tile_q", "decode", "kv_chunk", "max_chunks", "num_work")] + [
        ("d_page_ids", C.c_void_p), ("stream", C.c_void_p), ("metadata_bytes", C.c_int64)]


_P = C.c_void_p
_I32, _I64, _F32, _F64, _SZ = C.c_int32, C.c_int64, C.c_float, C.c_double, C.c_size_t


def _sig(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_plan = _sig("pg_plan_paged_prefill", C.c_int, C.POINTER(_P), _I32, _P, _P, _P, _P, _P,
             _I32, _I32, _I32, _I32, _P)
_plan_ring = _sig("pg_plan_paged_prefill_ring", C.c_int, C.POINTER(_P), _I32, _P, _P, _P, _P,
                  _I32, _I32, _I32, _I32, _I32, _P)
_plan_seg = _sig("pg_plan_paged_segment", C.c_int, C.POINTER(_P), _I32, _P, _P, _P, _P, _P, _P,
                 _I32, _I32, _I32, _I32, _P)
_destroy = _sig("pg_plan_destroy", None, _P)
_info = _sig("pg_plan_info", C.c_int, _P, C.POINTER(pg_plan_info_t))
_rope = _sig("pg_rope_table", C.c_int, _P, _P, _I32, _I32, _F64, _P)
_prep256 = _sig("pg_prep_paged_hd256", C.c_int, _P, C.POINTER(pg_pool_t), _I32,
                _P, _I64, _P, _I64, _P, _I64, _P, _P, _F32, _P, _P, _I32, _P, _P)
_prep512 = _sig("pg_prep_paged_hd512", C.c_int, _P, C.POINTER(pg_pool_t), _I32,
                _P, _I64, _P, _I64, _P, _P, _F32, _P, _P, _I32, _P, _P)
_wsb = _sig("pg_workspace_bytes", _SZ, _P)
_attn256 = _sig("pg_attn_paged_prefill", C.c_int, _P, C.POINTER(pg_pool_t), _I32, _P, _P,
                _I32, _F32, _P, _SZ, _P)
_attn512 = _sig("pg_attn_paged_prefill_hd512", C.c_int, _P, C.POINTER(pg_pool_t), _I32, _P, _P,
                _I32, _F32, _P, _SZ, _P)
_attn_noalloc = _sig("pg_attn_paged_decode_noalloc", C.c_int, _P, C.POINTER(pg_pool_t), _I32,
                    _P, _P, _I32, _F32, _P)
PG_NOALLOC_SCRATCH_BYTES = 32 << 20
_devstat = _sig("pg_device_status", C.c_int, _P)
_launches = _sig("pg_launch_count", _I64)
_test_wait = _sig("pg_test_bounded_wait", C.c_int, _I32, _I64)
_sstr = _sig("pg_status_string", C.c_char_p, C.c_int)


# ------------------------------------------------------------------------------ helpers
def _ptr(t) -> int | None:
    """Device address of a torch tensor (None passes NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _host(a, dtype):
    if a is None:
        return None, None
    arr = np.ascontiguousarray(np.asarray(a), dtype=dtype)
    return arr, arr.ctypes.data


def check(status: int, what: str = "pg call") -> None:
    if status != PG_OK:
        raise PgError(status, what)


def pg_status_string(status: int) -> str:
    return _sstr(int(status)).decode()


def pg_launch_count() -> int:
    return int(_launches())


def pg_test_bounded_wait(withhold, wait_limit_ns=0) -> int:
    """Test hook: withhold=1 makes later tensor-core prefill launches skip one key-tile
    arrival and give up their bounded waits after wait_limit_ns; withhold=0 restores them."""
    return int(_test_wait(int(withhold), int(wait_limit_ns)))


def pg_device_status(stream=None) -> int:
    return _devstat(_stream(stream))


# ------------------------------------------------------------------------------ plan
class Plan:
    """Owning handle of a ``pg_plan_t``; destroyed with the object or ``close()``."""

    def __init__(self, handle: int):
        self.handle = handle

    def close(self):
        if self.handle:
            _destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def info(self) -> pg_plan_info_t:
        i = pg_plan_info_t()
        check(_info(self.handle, C.byref(i)), "pg_plan_info")
        return i

    @property
    def _as_parameter_(self):
        return self.handle


def pg_plan_paged_prefill(plan, num_req, qo_indptr, kv_page_indptr, page_ids, last_page_len,
                          start_pos, num_qo_heads, num_kv_heads, head_dim, page_size,
                          stream=None):
    """Build (plan=None) or update (plan=Plan) a plan. Returns (status, Plan or None)."""
    h = _P(plan.handle if plan is not None else None)
    keep = [_host(qo_indptr, np.int64), _host(kv_page_indptr, np.int64),
            _host(page_ids, np.int32), _host(last_page_len, np.int32), _host(start_pos, np.int64)]
    rc = _plan(C.byref(h), int(num_req), *[k[1] for k in keep], int(num_qo_heads),
               int(num_kv_heads), int(head_dim), int(page_size), _stream(stream))
    del keep
    if plan is not None:
        return rc, plan
    return rc, (Plan(h.value) if rc == PG_OK else None)


def pg_plan_paged_prefill_ring(plan, num_req, qo_indptr, kv_page_indptr, page_ids, start_pos,
                               num_qo_heads, num_kv_heads, head_dim, page_size, window_left,
                               stream=None):
    """Build (plan=None) or update (plan=Plan) a ring-addressed plan. Returns (status, Plan
    or None)."""
    h = _P(plan.handle if plan is not None else None)
    keep = [_host(qo_indptr, np.int64), _host(kv_page_indptr, np.int64),
            _host(page_ids, np.int32), _host(start_pos, np.int64)]
    rc = _plan_ring(C.byref(h), int(num_req), *[k[1] for k in keep], int(num_qo_heads),
                    int(num_kv_heads), int(head_dim), int(page_size), int(window_left),
                    _stream(stream))
    del keep
    if plan is not None:
        return rc, plan
    return rc, (Plan(h.value) if rc == PG_OK else None)


def pg_plan_paged_segment(plan, num_req, qo_indptr, kv_page_indptr, page_ids, last_page_len,
                          kv_start, start_pos, num_qo_heads, num_kv_heads, head_dim, page_size,
                          stream=None):
    """Build (plan=None) or update (plan=Plan) a key-segment plan. Returns (status, Plan or
    None)."""
    h = _P(plan.handle if plan is not None else None)
    keep = [_host(qo_indptr, np.int64), _host(kv_page_indptr, np.int64),
            _host(page_ids, np.int32), _host(last_page_len, np.int32),
            _host(kv_start, np.int64), _host(start_pos, np.int64)]
    rc = _plan_seg(C.byref(h), int(num_req), *[k[1] for k in keep], int(num_qo_heads),
                   int(num_kv_heads), int(head_dim), int(page_size), _stream(stream))
    del keep
    if plan is not None:
        return rc, plan
    return rc, (Plan(h.value) if rc == PG_OK else None)


def pg_workspace_bytes(plan) -> int:
    return int(_wsb(plan.handle if plan is not None else None))


# ------------------------------------------------------------------------------ pool
def pool_descriptor(pool, **override) -> pg_pool_t:
    """pg_pool_t for a torch bf16 tensor shaped [L, P, 2, Hkv, ps, D] (strides taken from the
    tensor, so a non-dense tensor is reported by the library, not hidden here)."""
    L, P, two, Hkv, ps, D = pool.shape
    st = pool.stride()
    d = pg_pool_t(pool.data_ptr(), L, P, ps, Hkv, D, st[0], st[1], st[2], st[3], st[4],
                  pool.numel())
    for k, v in override.items():
        setattr(d, k, v)
    return d


# ------------------------------------------------------------------------------ kernels
def pg_rope_table(rope_cos, rope_sin, rows, head_dim, theta, stream=None) -> int:
    return _rope(_ptr(rope_cos), _ptr(rope_sin), int(rows), int(head_dim), float(theta),
                 _stream(stream))


def pg_prep_paged_hd256(plan, pool: pg_pool_t, layer, q_raw, q_tok_stride, k_raw, k_tok_stride,
                        v_raw, v_tok_stride, w_q, w_k, eps, rope_cos, rope_sin, rope_rows,
                        q_out, stream=None) -> int:
    return _prep256(plan.handle if plan is not None else None, C.byref(pool), int(layer),
                    _ptr(q_raw), int(q_tok_stride), _ptr(k_raw), int(k_tok_stride), _ptr(v_raw),
                    int(v_tok_stride), _ptr(w_q), _ptr(w_k), float(eps), _ptr(rope_cos),
                    _ptr(rope_sin), int(rope_rows), _ptr(q_out), _stream(stream))


def pg_prep_paged_hd512(plan, pool: pg_pool_t, layer, q_raw, q_tok_stride, k_raw, k_tok_stride,
                        w_q, w_k, eps, rope_cos, rope_sin, rope_rows, q_out,
                        stream=None) -> int:
    return _prep512(plan.handle if plan is not None else None, C.byref(pool), int(layer),
                    _ptr(q_raw), int(q_tok_stride), _ptr(k_raw), int(k_tok_stride), _ptr(w_q),
                    _ptr(w_k), float(eps), _ptr(rope_cos), _ptr(rope_sin), int(rope_rows),
                    _ptr(q_out), _stream(stream))


def pg_attn_paged_prefill(plan, pool: pg_pool_t, layer, q, out, window_left, sm_scale,
                          workspace=None, ws_bytes=0, stream=None) -> int:
    return _attn256(plan.handle if plan is not None else None, C.byref(pool), int(layer), _ptr(q),
                    _ptr(out), int(window_left), float(sm_scale), _ptr(workspace), int(ws_bytes),
                    _stream(stream))


def pg_attn_paged_prefill_hd512(plan, pool: pg_pool_t, layer, q, out, window_left, sm_scale,
                                workspace=None, ws_bytes=0, stream=None) -> int:
    return _attn512(plan.handle if plan is not None else None, C.byref(pool), int(layer), _ptr(q),
                    _ptr(out), int(window_left), float(sm_scale), _ptr(workspace), int(ws_bytes),
                    _stream(stream))


_attn256_lse = _sig("pg_attn_paged_prefill_lse", C.c_int, _P, C.POINTER(pg_pool_t), _I32, _P, _P,
                    _P, _I32, _F32, _P, C.c_size_t, _P)
_attn512_lse = _sig("pg_attn_paged_prefill_hd512_lse", C.c_int, _P, C.POINTER(pg_pool_t), _I32, _P,
                    _P, _P, _I32, _F32, _P, C.c_size_t, _P)
_merge = _sig("pg_merge_attn_states", C.c_int, _P, _P, _P, _P, _P, _P, _I64, _I32, _P)


def pg_attn_paged_prefill_lse(plan, pool: pg_pool_t, layer, q, out, lse, window_left, sm_scale,
                              workspace=None, ws_bytes=0, stream=None) -> int:
    return _attn256_lse(plan.handle if plan is not None else None, C.byref(pool), int(layer),
                        _ptr(q), _ptr(out), _ptr(lse), int(window_left), float(sm_scale),
                        _ptr(workspace), int(ws_bytes), _stream(stream))


def pg_attn_paged_prefill_hd512_lse(plan, pool: pg_pool_t, layer, q, out, lse, window_left,
                                    sm_scale, workspace=None, ws_bytes=0, stream=None) -> int:
    return _attn512_lse(plan.handle if plan is not None else None, C.byref(pool), int(layer),
                        _ptr(q), _ptr(out), _ptr(lse), int(window_left), float(sm_scale),
                        _ptr(workspace), int(ws_bytes), _stream(stream))


def pg_merge_attn_states(out_a, lse_a, out_b, lse_b, out, lse, rows, head_dim,
                         stream=None) -> int:
    return _merge(_ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b), _ptr(out), _ptr(lse),
                  int(rows), int(head_dim), _stream(stream))


def pg_attn_paged_decode_noalloc(plan, pool: pg_pool_t, layer, q, out, window_left, sm_scale,
                                 stream=None) -> int:
    """Decode attention with the library's static scratch; allocates nothing."""
    return _attn_noalloc(plan.handle if plan is not None else None, C.byref(pool), int(layer),
                         _ptr(q), _ptr(out), int(window_left), float(sm_scale), _stream(stream))


EXPORTED = ["pg_plan_paged_prefill", "pg_plan_paged_prefill_ring", "pg_plan_paged_segment",
            "pg_attn_paged_prefill_lse", "pg_attn_paged_prefill_hd512_lse", "pg_merge_attn_states",
            "pg_plan_destroy", "pg_plan_info", "pg_rope_table",
            "pg_prep_paged_hd256", "pg_prep_paged_hd512", "pg_workspace_bytes",
            "pg_attn_paged_prefill", "pg_attn_paged_prefill_hd512", "pg_device_status",
            "pg_launch_count", "pg_status_string", "pg_test_bounded_wait"]


# ---------------------------------------------------------------- page accounting (include/pg_kv.h)
PG_KV_OK = 0
PG_KV_ERR_ARG = -101
PG_KV_ERR_NO_PAGES = -102
PG_KV_ERR_WINDOW = -103
PG_KV_ERR_ROPE = -104
PG_KV_ERR_FOREIGN = -105
PG_KV_ERR_FRONTIER = -106
PG_KV_ERR_CAPACITY = -107
PG_KV_ERR_PENDING = -108
PG_KV_LOCAL = 0
PG_KV_GLOBAL = 1

_I32P, _I64P = C.POINTER(C.c_int32), C.POINTER(C.c_int64)
_lib.pg_kv_server_create.argtypes = [C.POINTER(C.c_void_p), C.c_int32, C.c_int32, C.c_int32,
                                     C.c_int32, C.c_int32, C.c_int32]
_lib.pg_kv_server_destroy.argtypes = [C.c_void_p]
_lib.pg_kv_server_destroy.restype = None
_lib.pg_kv_request_open.argtypes = [C.c_void_p, _I64P]
_lib.pg_kv_request_close.argtypes = [C.c_void_p, C.c_int64]
_lib.pg_kv_admit_step.argtypes = [C.c_void_p, C.c_int64, C.c_int32]
_lib.pg_kv_commit_step.argtypes = [C.c_void_p, C.c_int64]
_lib.pg_kv_abort_step.argtypes = [C.c_void_p, C.c_int64]
_lib.pg_kv_request_pending.argtypes = [C.c_void_p, C.c_int64, _I32P]
_lib.pg_kv_request_info.argtypes = [C.c_void_p, C.c_int64, _I32P, _I32P, _I32P]
_lib.pg_kv_request_pages.argtypes = [C.c_void_p, C.c_int64, C.c_int32, C.c_void_p, C.c_int32, _I32P]
_lib.pg_kv_free_pages.argtypes = [C.c_void_p, C.c_int32, _I32P]
_lib.pg_kv_inject_refusal.argtypes = [C.c_void_p, C.c_int32, C.c_int32]
_lib.pg_kv_batch_plan_inputs.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                         C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p,
                                         _I32P]


def pg_kv_server_create(pages_local, pages_global, page_size, window_left, fail_closed_at_window,
                        rope_rows):
    """Returns (status, server handle or None)."""
    h = C.c_void_p()
    rc = _lib.pg_kv_server_create(C.byref(h), int(pages_local), int(pages_global), int(page_size),
                                  int(window_left), int(fail_closed_at_window), int(rope_rows))
    return rc, (h if rc == PG_KV_OK else None)


_lib.pg_kv_server_create_ring.argtypes = [C.POINTER(C.c_void_p), C.c_int32, C.c_int32, C.c_int32,
                                          C.c_int32, C.c_int32, C.c_int32]
_lib.pg_kv_server_create_ring.restype = C.c_int


def pg_kv_server_create_ring(pages_local, pages_global, page_size, window_left, ring_max_step,
                             rope_rows):
    """Server whose local family keeps a ring of pages. Returns (status, handle or None)."""
    h = C.c_void_p()
    rc = _lib.pg_kv_server_create_ring(C.byref(h), int(pages_local), int(pages_global),
                                       int(page_size), int(window_left), int(ring_max_step),
                                       int(rope_rows))
    return rc, (h if rc == PG_KV_OK else None)


def pg_kv_server_destroy(srv) -> None:
    _lib.pg_kv_server_destroy(srv)


def pg_kv_request_open(srv):
    """Returns (status, request id)."""
    rid = C.c_int64()
    rc = _lib.pg_kv_request_open(srv, C.byref(rid))
    return rc, rid.value


def pg_kv_request_close(srv, request_id) -> int:
    return _lib.pg_kv_request_close(srv, int(request_id))


def pg_kv_admit_step(srv, request_id, n_tokens) -> int:
    return _lib.pg_kv_admit_step(srv, int(request_id), int(n_tokens))


def pg_kv_commit_step(srv, request_id) -> int:
    return _lib.pg_kv_commit_step(srv, int(request_id))


def pg_kv_abort_step(srv, request_id) -> int:
    return _lib.pg_kv_abort_step(srv, int(request_id))


def pg_kv_request_pending(srv, request_id):
    """Returns (status, tokens of the pending step, 0 when none)."""
    n = C.c_int32()
    rc = _lib.pg_kv_request_pending(srv, int(request_id), C.byref(n))
    return rc, n.value


def pg_kv_request_info(srv, request_id):
    """Returns (status, frontier, pages_local, pages_global)."""
    f, pl, pg_ = C.c_int32(), C.c_int32(), C.c_int32()
    rc = _lib.pg_kv_request_info(srv, int(request_id), C.byref(f), C.byref(pl), C.byref(pg_))
    return rc, f.value, pl.value, pg_.value


def pg_kv_request_pages(srv, request_id, family, cap=1 << 20):
    """Returns (status, int32 array of page ids)."""
    out = np.empty(max(cap, 1), np.int32)
    n = C.c_int32()
    rc = _lib.pg_kv_request_pages(srv, int(request_id), int(family), out.ctypes.data, int(cap),
                                  C.byref(n))
    return rc, out[:n.value].copy() if rc == PG_KV_OK else None


def pg_kv_free_pages(srv, family):
    """Returns (status, free page count)."""
    n = C.c_int32()
    rc = _lib.pg_kv_free_pages(srv, int(family), C.byref(n))
    return rc, n.value


def pg_kv_inject_refusal(srv, family, count) -> int:
    return _lib.pg_kv_inject_refusal(srv, int(family), int(count))


def pg_kv_batch_plan_inputs(srv, family, request_ids, step_tokens, cap=1 << 20):
    """Returns (status, kv_page_indptr, page_ids, last_page_len, start_pos) as numpy arrays in
    pg_plan_paged_prefill's layout."""
    rids = np.ascontiguousarray(request_ids, np.int64)
    steps = np.ascontiguousarray(step_tokens, np.int32)
    n = len(rids)
    indptr = np.zeros(n + 1, np.int64)
    pages = np.empty(max(cap, 1), np.int32)
    last = np.zeros(max(n, 1), np.int32)
    start = np.zeros(max(n, 1), np.int64)
    cnt = C.c_int32()
    rc = _lib.pg_kv_batch_plan_inputs(srv, int(family), n, rids.ctypes.data, steps.ctypes.data,
                                      indptr.ctypes.data, pages.ctypes.data, int(cap),
                                      last.ctypes.data, start.ctypes.data, C.byref(cnt))
    if rc != PG_KV_OK:
        return rc, None, None, None, None
    return rc, indptr, pages[:cnt.value].copy(), last[:n].copy(), start[:n].copy()


EXPORTED += ["pg_kv_server_create", "pg_kv_server_create_ring", "pg_kv_server_destroy", "pg_kv_request_open",
             "pg_kv_request_close", "pg_kv_admit_step", "pg_kv_commit_step", "pg_kv_abort_step",
             "pg_kv_request_pending", "pg_kv_request_info", "pg_kv_request_pages",
             "pg_kv_free_pages", "pg_kv_inject_refusal", "pg_kv_batch_plan_inputs"]
