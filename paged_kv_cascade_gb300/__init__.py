"""Python binding of libpkc (paged-KV cascade decode attention for GB300).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libpkc.so``.  torch tensors supply device memory and the
current CUDA stream; their data pointers go straight to the C ABI declared
in ``include/pkc.h``.  If the library has not been built, every call raises
-- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpkc.so")

PKC_OK = 0
STATUS_NAMES = {0: "PKC_OK", 1: "PKC_ERR_INVALID_ARG", 2: "PKC_ERR_UNSUPPORTED",
                3: "PKC_ERR_WORKSPACE", 4: "PKC_ERR_BLOCK_TABLE", 5: "PKC_ERR_CUDA",
                6: "PKC_ERR_TIMEOUT", 7: "PKC_ERR_PLAN"}
F32, F16, BF16, E4M3 = 0, 1, 2, 3

# Header indices of the plan buffer (include/pkc.h).
PLAN_FIELDS = ["MAGIC", "TOTAL_WORDS", "NUM_CTAS", "TILE_Q", "N_REQ", "KV_CHUNK",
               "N_UNITS", "N_WORK", "N_PARTIALS", "N_SPLIT", "N_EMPTY",
               "OFF_CTA_INDPTR", "OFF_CTA_WORK", "OFF_WORK_UNIT", "OFF_WORK_KV_BEGIN",
               "OFF_WORK_KV_END", "OFF_WORK_PARTIAL", "OFF_UNIT_REQ", "OFF_UNIT_QTILE",
               "OFF_UNIT_KV_LEN", "OFF_UNIT_N_CHUNKS", "OFF_UNIT_PARTIAL_BEGIN",
               "OFF_UNIT_LIST", "OFF_CTA_COST", "OFF_WORK_ORDER", "OFF_ORDER_REC"]
PLAN = {name: i for i, name in enumerate(PLAN_FIELDS)}
PLAN_MAGIC = 0x504B4331

# Every symbol the C ABI exports, with (restype, argtypes).
_c = ctypes
_P, _I, _I64, _SZ, _F, _D = _c.c_void_p, _c.c_int, _c.c_int64, _c.c_size_t, _c.c_float, _c.c_double
SIGNATURES = {
    "pkc_version": (_I, []),
    "pkc_last_error": (_c.c_char_p, []),
    "pkc_merge_state": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I, _I, _I, _P]),
    "pkc_merge_states": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _I, _P]),
    "pkc_merge_states_to": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _I, _I, _P]),
    "pkc_plan_words": (_I, [_P, _I, _I, _I, _c.POINTER(_SZ)]),
    "pkc_plan": (_I, [_P, _P, _I, _I, _I, _D, _D, _P, _SZ]),
    "pkc_plan_upload": (_I, [_P, _P, _SZ, _P]),
    "pkc_workspace_size": (_I, [_I, _I, _I, _I, _I, _c.POINTER(_SZ)]),
    "pkc_workspace_init": (_I, [_P, _SZ, _P]),
    "pkc_device_status": (_I, [_P, _P, _c.POINTER(_c.c_int32)]),
    "pkc_paged_decode_state": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I64, _F,
                                    _P, _P, _SZ, _P, _P, _I, _P]),
    "pkc_prefix_attention_state": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _SZ,
                                        _P, _P, _I, _P]),
    "pkc_paged_decode_state_noalloc": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I64,
                                            _F, _P, _P, _P, _P, _I, _P]),
    "pkc_paged_decode_state_fp8": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I64, _F,
                                        _F, _F, _P, _P, _SZ, _P, _P, _P]),
    "pkc_set_stage_events": (_I, [_c.POINTER(_P), _I]),
    "pkc_set_decode_kernel": (_I, [_I]),
    "pkc_set_decode_schedule": (_I, [_I]),
    "pkc_set_contraction": (_I, [_I]),
    "pkc_set_prefix_ctas": (_I, [_I]),
    "pkc_set_cascade_small": (_I, [_I]),
    "pkc_last_launch_blocks": (_I, [_c.POINTER(_c.c_int), _c.POINTER(_c.c_int)]),
    "pkc_selftest_wait_timeout": (_I, [_P, _SZ, _c.POINTER(_c.c_int32), _P]),
    "pkc_append_kv": (_I, [_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I64, _I, _P, _SZ, _P]),
    "pkc_cascade_decode_multilevel": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _I, _I, _I,
                                           _I, _I, _I64, _F, _P, _P, _SZ, _P, _P, _I, _P]),
    "pkc_cascade_decode_paged_prefix": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _I, _I,
                                             _I, _I, _I, _I64, _F, _P, _P, _SZ, _P, _P, _I, _P]),
    "pkc_cascade_decode": (_I, [_P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I,
                                _I64, _F, _P, _P, _SZ, _P, _P, _I, _P]),
    "pkc_cascade_decode_state": (_I, [_P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _I, _I, _I, _I,
                                      _I, _I64, _F, _P, _P, _SZ, _P, _P, _I, _P]),
}

_lib = None
_lock = threading.Lock()


class PkcError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


def lib():
    """The loaded libpkc.so.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libpkc.so not found at {LIB_PATH}; build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _check(rc):
    if rc != PKC_OK:
        raise PkcError(rc, lib().pkc_last_error().decode())


def _dtype_code(t) -> int:
    import torch
    return {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}[t.dtype]


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _host_i32(a):
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def _hptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


# ---------------------------------------------------------------------------
# Argument checks.  The C ABI takes raw pointers and sizes, so a tensor of the
# wrong dtype, shape or device would be read past its end; the binding
# checks every tensor against the sizes it passes down.
# ---------------------------------------------------------------------------

def _expect(name, t, dtypes, shape, device=None):
    """t must be a contiguous CUDA tensor of one of `dtypes` whose shape
    matches `shape` (None entries match any size) on `device`."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {list(dtypes)}")
    if len(t.shape) != len(shape) or any(w is not None and w != g for g, w in zip(t.shape, shape)):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)} (None = any)")
    if not t.is_cuda or (device is not None and t.device != device):
        raise ValueError(f"{name} must be on {device if device is not None else 'a CUDA device'}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_paged(q, k_cache, v_cache, block_table, cache_seqlens, workspace, o, lse, kv_dtypes):
    """The common tensors of the paged-decode and cascade calls."""
    import torch
    _expect("q", q, (torch.float16, torch.bfloat16), (None, None, None))
    B, Hq, D = q.shape
    dev = q.device
    _expect("k_cache", k_cache, kv_dtypes, (None, None, None, D), dev)
    _expect("v_cache", v_cache, (k_cache.dtype,), tuple(k_cache.shape), dev)
    _expect("block_table", block_table, (torch.int32,), (B, None), dev)
    _expect("cache_seqlens", cache_seqlens, (torch.int32,), (B,), dev)
    if workspace is not None:
        _expect("workspace", workspace, (torch.uint8,), (None,), dev)
    if o is not None:
        _expect("o", o, (q.dtype,), (B, Hq, D), dev)
    if lse is not None:
        _expect("lse", lse, (torch.float32,), (B, Hq), dev)


def _check_prefix(q, k_prefix, v_prefix, prefix_kv_indptr):
    """Contiguous shared prefixes [L, Hkv, D] of q's dtype, L >= the last indptr."""
    _expect("k_prefix", k_prefix, (q.dtype,), (None, None, q.shape[2]), q.device)
    _expect("v_prefix", v_prefix, (q.dtype,), tuple(k_prefix.shape), q.device)
    if len(prefix_kv_indptr) and int(prefix_kv_indptr[-1]) > k_prefix.shape[0]:
        raise ValueError("prefix_kv_indptr ends past the prefix tensors")


def version() -> int:
    return lib().pkc_version()


# ---------------------------------------------------------------------------
# Merge operator
# ---------------------------------------------------------------------------

def merge_state(v_a, s_a, v_b, s_b, v_out=None, s_out=None, stream=None):
    """(v_a, s_a) (+) (v_b, s_b); v [T, H, D], s [T, H] float32."""
    import torch
    _expect("v_a", v_a, (torch.float32, torch.float16, torch.bfloat16), (None, None, None))
    T, H, D = v_a.shape
    for name, t, dt, shp in (("s_a", s_a, torch.float32, (T, H)), ("v_b", v_b, v_a.dtype, (T, H, D)),
                             ("s_b", s_b, torch.float32, (T, H)), ("v_out", v_out, v_a.dtype, (T, H, D)),
                             ("s_out", s_out, torch.float32, (T, H))):
        if t is not None:
            _expect(name, t, (dt,), shp, v_a.device)
    v_out = torch.empty_like(v_a) if v_out is None else v_out
    s_out = torch.empty_like(s_a) if s_out is None else s_out
    _check(lib().pkc_merge_state(_ptr(v_a), _ptr(s_a), _ptr(v_b), _ptr(s_b), _ptr(v_out),
                                 _ptr(s_out), T, H, D, _dtype_code(v_a), _stream(stream)))
    return v_out, s_out


def merge_states(v, s, v_out=None, s_out=None, stream=None):
    """n-ary (+) over axis 1: v [T, n, H, D], s [T, n, H] -> [T, H, D], [T, H]."""
    import torch
    _expect("v", v, (torch.float32, torch.float16, torch.bfloat16), (None, None, None, None))
    T, n, H, D = v.shape
    _expect("s", s, (torch.float32,), (T, n, H), v.device)
    if v_out is not None:
        _expect("v_out", v_out, (v.dtype,), (T, H, D), v.device)
    if s_out is not None:
        _expect("s_out", s_out, (torch.float32,), (T, H), v.device)
    v_out = torch.empty((T, H, D), dtype=v.dtype, device=v.device) if v_out is None else v_out
    s_out = torch.empty((T, H), dtype=torch.float32, device=v.device) if s_out is None else s_out
    _check(lib().pkc_merge_states(_ptr(v), _ptr(s), _ptr(v_out), _ptr(s_out), T, n, H, D,
                                  _dtype_code(v), _stream(stream)))
    return v_out, s_out


def merge_states_to(v, s, out_dtype, v_out=None, s_out=None, stream=None):
    """n-ary (+) of float32 states v [T, n, H, D], s [T, n, H] into a result
    of out_dtype (torch.float16 / torch.bfloat16 / torch.float32), rounded
    once."""
    import torch
    _expect("v", v, (torch.float32,), (None, None, None, None))
    T, n, H, D = v.shape
    _expect("s", s, (torch.float32,), (T, n, H), v.device)
    if v_out is not None:
        _expect("v_out", v_out, (out_dtype,), (T, H, D), v.device)
    if s_out is not None:
        _expect("s_out", s_out, (torch.float32,), (T, H), v.device)
    v_out = torch.empty((T, H, D), dtype=out_dtype, device=v.device) if v_out is None else v_out
    s_out = torch.empty((T, H), dtype=torch.float32, device=v.device) if s_out is None else s_out
    _check(lib().pkc_merge_states_to(_ptr(v), _ptr(s), _ptr(v_out), _ptr(s_out), T, n, H, D, F32,
                                     _dtype_code(v_out), _stream(stream)))
    return v_out, s_out


# ---------------------------------------------------------------------------
# Plan and workspace
# ---------------------------------------------------------------------------

def plan_words(n, num_ctas, tile_q=1, qo_len=None) -> int:
    q = None if qo_len is None else _host_i32(qo_len)
    out = ctypes.c_size_t()
    _check(lib().pkc_plan_words(_hptr(q), n, tile_q, num_ctas, ctypes.byref(out)))
    return out.value


def plan(kv_len, num_ctas, tile_q=1, qo_len=None, alpha=1.0, beta=1.0, out=None):
    """Host-side load-balanced plan; returns the int32 plan buffer."""
    kv = _host_i32(kv_len)
    q = None if qo_len is None else _host_i32(qo_len)
    words = plan_words(len(kv), num_ctas, tile_q, q)
    if out is None:
        out = np.zeros(words, np.int32)
    assert out.dtype == np.int32 and out.flags.c_contiguous and out.size >= words
    _check(lib().pkc_plan(_hptr(q), _hptr(kv), len(kv), tile_q, num_ctas, float(alpha),
                          float(beta), _hptr(out), out.size))
    return out


def plan_upload(plan_buf, workspace, stream=None):
    _check(lib().pkc_plan_upload(_hptr(plan_buf), _ptr(workspace), workspace.numel(),
                                 _stream(stream)))


def workspace_size(batch, num_qo_heads, num_ctas=0, prefix_splits=0, head_dim=128) -> int:
    out = ctypes.c_size_t()
    _check(lib().pkc_workspace_size(batch, num_qo_heads, head_dim, num_ctas, prefix_splits,
                                    ctypes.byref(out)))
    return out.value


def workspace_init(workspace, stream=None):
    _check(lib().pkc_workspace_init(_ptr(workspace), workspace.numel(), _stream(stream)))


def device_status(workspace, stream=None) -> int:
    st = ctypes.c_int32()
    _check(lib().pkc_device_status(_ptr(workspace), _stream(stream), ctypes.byref(st)))
    return st.value


# ---------------------------------------------------------------------------
# Attention states
# ---------------------------------------------------------------------------

def paged_decode_state(q, k_cache, v_cache, block_table, cache_seqlens, sm_scale, workspace,
                       plan_buf=None, o=None, lse=None, stream=None):
    """States of q [B, Hq, 128] over each request's paged cache."""
    import torch
    _check_paged(q, k_cache, v_cache, block_table, cache_seqlens, workspace, o, lse, (q.dtype,))
    B, Hq, D = q.shape
    P, ps, Hkv, _ = k_cache.shape
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib().pkc_paged_decode_state(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(cache_seqlens), B, Hq, Hkv, D, ps, P, float(sm_scale), _hptr(plan_buf),
        _ptr(workspace), workspace.numel(), _ptr(o), _ptr(lse), _dtype_code(q), _stream(stream)))
    return o, lse


def paged_decode_state_fp8(q, k_cache, v_cache, block_table, cache_seqlens, sm_scale, workspace,
                           k_scale=1.0, v_scale=1.0, plan_buf=None, o=None, lse=None, stream=None):
    """States of fp16 q [B, Hq, 128] over an e4m3 paged cache (uint8 codes
    [P, page_size, Hkv, 128]); the cached values are k_scale * e4m3(k) and
    v_scale * e4m3(v)."""
    import torch
    B, Hq, D = q.shape
    P, ps, Hkv, _ = k_cache.shape
    if q.dtype != torch.float16 or k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise TypeError("paged_decode_state_fp8: q must be float16 and the caches uint8 e4m3 codes")
    _check_paged(q, k_cache, v_cache, block_table, cache_seqlens, workspace, o, lse, (torch.uint8,))
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib().pkc_paged_decode_state_fp8(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(cache_seqlens), B, Hq, Hkv, D, ps, P, float(sm_scale), float(k_scale), float(v_scale),
        _hptr(plan_buf), _ptr(workspace), workspace.numel(), _ptr(o), _ptr(lse), _stream(stream)))
    return o, lse


def append_kv(k_new, v_new, k_cache, v_cache, block_table, cache_seqlens, workspace,
              append_mask=None, stream=None):
    """Write one new token per request (k_new / v_new [B, Hkv, 128]) into the
    paged cache at each request's next slot and grow cache_seqlens by one, in
    place; an fp8 cache takes uint8 e4m3 codes."""
    import torch
    _expect("k_cache", k_cache, (torch.float16, torch.bfloat16, torch.uint8), (None, None, None, None))
    P, ps, Hkv, D = k_cache.shape
    dev = k_cache.device
    _expect("v_cache", v_cache, (k_cache.dtype,), tuple(k_cache.shape), dev)
    _expect("k_new", k_new, (k_cache.dtype,), (None, Hkv, D), dev)
    B = k_new.shape[0]
    _expect("v_new", v_new, (k_cache.dtype,), (B, Hkv, D), dev)
    _expect("block_table", block_table, (torch.int32,), (B, None), dev)
    _expect("cache_seqlens", cache_seqlens, (torch.int32,), (B,), dev)
    _expect("workspace", workspace, (torch.uint8,), (None,), dev)
    if append_mask is not None:
        _expect("append_mask", append_mask, (torch.uint8,), (B,), dev)
    if k_cache.dtype == torch.uint8:
        code = E4M3
    else:
        code = _dtype_code(k_cache)
    _check(lib().pkc_append_kv(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], _ptr(cache_seqlens), _ptr(append_mask), B, Hkv, D, ps, P, code,
        _ptr(workspace), workspace.numel(), _stream(stream)))


DECODE_KERNELS = {"auto": 0, "simt": 1, "mma": 2}


def set_decode_kernel(which):
    """Kernel for 16-bit paged decode: "auto", "simt" (CUDA cores) or "mma"
    (tensor cores); process-wide."""
    _check(lib().pkc_set_decode_kernel(DECODE_KERNELS[which]))


DECODE_SCHEDULES = {"dynamic": 1, "static": 0}


def set_decode_schedule(which):
    """Schedule of a planned decode: "dynamic" (blocks take the plan's chunks
    from a shared longest-first queue; default) or "static" (each block runs
    its CTA's list of the plan); process-wide."""
    _check(lib().pkc_set_decode_schedule(DECODE_SCHEDULES[which]))


def set_contraction(which):
    """'separate' (default): a standalone contraction kernel, launched as the
    suffix decode's programmatic dependent; 'separate_plain': the same kernel
    launched plainly; 'fused': the attention kernels contract split states
    themselves (one launch fewer).  All give the same bits."""
    _check(lib().pkc_set_contraction({"separate": 0, "fused": 1, "separate_plain": 2}[which]))


def set_cascade_small(max_rows):
    """Largest query rows per KV head of a prefix group for which an unplanned
    cascade reads its prefixes through the decode kernel (one launch); 0 never."""
    _check(lib().pkc_set_cascade_small(int(max_rows)))


def set_prefix_ctas(n):
    """Thread blocks of the prefix stage: n > 0 caps them at n; 0 (default)
    is automatic: every SM, or, in a planned cascade call whose prefix is
    bound by the tensor pipe, a quarter of the SMs next to a dynamically
    scheduled decode on the rest (pkc.h, pkc_set_prefix_ctas); process-wide."""
    n = int(n)
    if n < 0:
        raise ValueError(f"set_prefix_ctas: n must be >= 0 (got {n})")
    _check(lib().pkc_set_prefix_ctas(n))


def last_launch_blocks():
    """(prefix blocks, decode blocks) of this thread's last cascade call."""
    pb, db = _c.c_int(0), _c.c_int(0)
    _check(lib().pkc_last_launch_blocks(_c.byref(pb), _c.byref(db)))
    return pb.value, db.value


def paged_decode_state_noalloc(q, k_cache, v_cache, block_table, cache_seqlens, sm_scale,
                               plan_buf=None, o=None, lse=None, device_status=None, stream=None):
    """paged_decode_state without a caller workspace, for callers that
    cannot allocate device memory: the library's own fixed 8 MiB device
    array holds the scratch.  Calls that overlap on the GPU race on it."""
    import torch
    _check_paged(q, k_cache, v_cache, block_table, cache_seqlens, None, o, lse, (q.dtype,))
    B, Hq, D = q.shape
    P, ps, Hkv, _ = k_cache.shape
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib().pkc_paged_decode_state_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(cache_seqlens), B, Hq, Hkv, D, ps, P, float(sm_scale), _hptr(plan_buf), _ptr(o),
        _ptr(lse), _ptr(device_status), _dtype_code(q), _stream(stream)))
    return o, lse


def prefix_attention_state(q, k_prefix, v_prefix, prefix_kv_indptr, prefix_req_indptr, sm_scale,
                           workspace, o=None, lse=None, stream=None):
    """States of q [B, Hq, 128] over each request's shared prefix (fp32 O)."""
    import torch
    _expect("q", q, (torch.float16, torch.bfloat16), (None, None, None))
    _check_prefix(q, k_prefix, v_prefix, _host_i32(prefix_kv_indptr))
    _expect("workspace", workspace, (torch.uint8,), (None,), q.device)
    if o is not None:
        _expect("o", o, (torch.float32,), tuple(q.shape), q.device)
    if lse is not None:
        _expect("lse", lse, (torch.float32,), tuple(q.shape[:2]), q.device)
    B, Hq, D = q.shape
    Hkv = k_prefix.shape[1]
    kv_ptr, req_ptr = _host_i32(prefix_kv_indptr), _host_i32(prefix_req_indptr)
    o = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device) if o is None else o
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib().pkc_prefix_attention_state(
        _ptr(q), _ptr(k_prefix), _ptr(v_prefix), _hptr(kv_ptr), _hptr(req_ptr), len(kv_ptr) - 1,
        B, Hq, Hkv, D, float(sm_scale), _ptr(workspace), workspace.numel(), _ptr(o), _ptr(lse),
        _dtype_code(q), _stream(stream)))
    return o, lse


def cascade_decode(q, k_prefix, v_prefix, prefix_kv_indptr, prefix_req_indptr, k_cache, v_cache,
                   block_table, cache_seqlens, sm_scale, workspace, plan_buf=None, o=None,
                   lse=None, stream=None):
    """Final O [B, Hq, 128] and LSE [B, Hq] over shared prefix + paged suffix."""
    import torch
    _check_paged(q, k_cache, v_cache, block_table, cache_seqlens, workspace, o, lse, (q.dtype,))
    _check_prefix(q, k_prefix, v_prefix, _host_i32(prefix_kv_indptr))
    B, Hq, D = q.shape
    P, ps, Hkv, _ = k_cache.shape
    kv_ptr, req_ptr = _host_i32(prefix_kv_indptr), _host_i32(prefix_req_indptr)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib().pkc_cascade_decode(
        _ptr(q), _ptr(k_prefix), _ptr(v_prefix), _hptr(kv_ptr), _hptr(req_ptr), len(kv_ptr) - 1,
        _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1], _ptr(cache_seqlens),
        B, Hq, Hkv, D, ps, P, float(sm_scale), _hptr(plan_buf), _ptr(workspace),
        workspace.numel(), _ptr(o), _ptr(lse), _dtype_code(q), _stream(stream)))
    return o, lse


def cascade_decode_state(q, k_prefix, v_prefix, prefix_kv_indptr, prefix_req_indptr, k_cache,
                         v_cache, block_table, cache_seqlens, sm_scale, workspace, plan_buf=None,
                         o=None, lse=None, stream=None):
    """cascade_decode returning the unrounded state: O [B, Hq, 128] float32 and
    LSE [B, Hq], for states merged further (KV sharding)."""
    import torch
    B, Hq, D = q.shape
    _check_paged(q, k_cache, v_cache, block_table, cache_seqlens, workspace, None, lse, (q.dtype,))
    _check_prefix(q, k_prefix, v_prefix, _host_i32(prefix_kv_indptr))
    if o is not None:
        _expect("o", o, (torch.float32,), (B, Hq, D), q.device)
    P, ps, Hkv, _ = k_cache.shape
    kv_ptr, req_ptr = _host_i32(prefix_kv_indptr), _host_i32(prefix_req_indptr)
    o = torch.empty((B, Hq, D), dtype=torch.float32, device=q.device) if o is None else o
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib().pkc_cascade_decode_state(
        _ptr(q), _ptr(k_prefix), _ptr(v_prefix), _hptr(kv_ptr), _hptr(req_ptr), len(kv_ptr) - 1,
        _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1], _ptr(cache_seqlens),
        B, Hq, Hkv, D, ps, P, float(sm_scale), _hptr(plan_buf), _ptr(workspace),
        workspace.numel(), _ptr(o), _ptr(lse), _dtype_code(q), _stream(stream)))
    return o, lse


def cascade_decode_multilevel(q, k_prefix, v_prefix, prefix_kv_indptr, prefix_req_ranges, k_cache,
                              v_cache, block_table, cache_seqlens, sm_scale, workspace, plan_buf=None,
                              o=None, lse=None, stream=None):
    """The cascade with prefix groups as request ranges [(begin, end)] that may
    overlap: each request attends to every group's prefix that holds it."""
    import torch
    _check_paged(q, k_cache, v_cache, block_table, cache_seqlens, workspace, o, lse, (q.dtype,))
    _check_prefix(q, k_prefix, v_prefix, _host_i32(prefix_kv_indptr))
    B, Hq, D = q.shape
    P, ps, Hkv, _ = k_cache.shape
    kv_ptr = _host_i32(prefix_kv_indptr)
    rr = _host_i32(prefix_req_ranges).reshape(-1, 2)
    rb, re = np.ascontiguousarray(rr[:, 0]), np.ascontiguousarray(rr[:, 1])
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib().pkc_cascade_decode_multilevel(
        _ptr(q), _ptr(k_prefix), _ptr(v_prefix), _hptr(kv_ptr), _hptr(rb), _hptr(re), len(kv_ptr) - 1,
        _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1], _ptr(cache_seqlens),
        B, Hq, Hkv, D, ps, P, float(sm_scale), _hptr(plan_buf), _ptr(workspace),
        workspace.numel(), _ptr(o), _ptr(lse), _dtype_code(q), _stream(stream)))
    return o, lse


def cascade_decode_paged_prefix(q, prefix_pages, prefix_page_indptr, prefix_kv_indptr,
                                prefix_req_ranges, k_cache, v_cache, block_table, cache_seqlens,
                                sm_scale, workspace, plan_buf=None, o=None, lse=None, stream=None):
    """The multi-level cascade with each group's prefix read in place from the
    page pool: prefix_pages (device int32) lists group j's pages at
    prefix_page_indptr[j] .. prefix_page_indptr[j+1]-1."""
    import torch
    _check_paged(q, k_cache, v_cache, block_table, cache_seqlens, workspace, o, lse, (q.dtype,))
    _expect("prefix_pages", prefix_pages, (torch.int32,), (None,), q.device)
    if len(prefix_page_indptr) and int(_host_i32(prefix_page_indptr)[-1]) > prefix_pages.shape[0]:
        raise ValueError("prefix_page_indptr ends past prefix_pages")
    B, Hq, D = q.shape
    P, ps, Hkv, _ = k_cache.shape
    kv_ptr, pg_ptr = _host_i32(prefix_kv_indptr), _host_i32(prefix_page_indptr)
    rr = _host_i32(prefix_req_ranges).reshape(-1, 2)
    rb, re = np.ascontiguousarray(rr[:, 0]), np.ascontiguousarray(rr[:, 1])
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib().pkc_cascade_decode_paged_prefix(
        _ptr(q), _ptr(prefix_pages), _hptr(pg_ptr), _hptr(kv_ptr), _hptr(rb), _hptr(re), len(kv_ptr) - 1,
        _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1], _ptr(cache_seqlens),
        B, Hq, Hkv, D, ps, P, float(sm_scale), _hptr(plan_buf), _ptr(workspace),
        workspace.numel(), _ptr(o), _ptr(lse), _dtype_code(q), _stream(stream)))
    return o, lse


def selftest_wait_timeout(workspace, stream=None) -> bool:
    """Run the bounded-wait failure path on the GPU (about 2 s): True if the
    wait gave up and returned as designed; the status word then holds
    PKC_ERR_TIMEOUT (read it with device_status)."""
    import torch
    _expect("workspace", workspace, (torch.uint8,), (None,))
    out = ctypes.c_int32(0)
    _check(lib().pkc_selftest_wait_timeout(_ptr(workspace), workspace.numel(), ctypes.byref(out),
                                           _stream(stream)))
    return out.value == 1


def set_stage_events(events):
    """Record 4 torch.cuda.Event objects around the stages of the next
    cascade_decode call on this thread (None clears)."""
    if events is None:
        _check(lib().pkc_set_stage_events(None, 0))
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib().pkc_set_stage_events(arr, len(events)))


def plan_dict(buf):
    """Decode a plan buffer into Python lists (for inspection and tests)."""
    h = {k: int(buf[v]) for k, v in PLAN.items()}
    nc, nw, nu = h["NUM_CTAS"], h["N_WORK"], h["N_UNITS"]

    def arr(off, n):
        return buf[h[off]:h[off] + n].tolist()
    indptr = arr("OFF_CTA_INDPTR", nc + 1)
    cta_work_flat = arr("OFF_CTA_WORK", nw)
    return {
        "header": h,
        "kv_chunk": h["KV_CHUNK"],
        "cta_work": [cta_work_flat[indptr[c]:indptr[c + 1]] for c in range(nc)],
        "work": list(zip(arr("OFF_WORK_UNIT", nw), arr("OFF_WORK_KV_BEGIN", nw),
                         arr("OFF_WORK_KV_END", nw))),
        "partial": arr("OFF_WORK_PARTIAL", nw),
        "unit_req": arr("OFF_UNIT_REQ", nu),
        "unit_qtile": arr("OFF_UNIT_QTILE", nu),
        "unit_kv_len": arr("OFF_UNIT_KV_LEN", nu),
        "unit_n_chunks": arr("OFF_UNIT_N_CHUNKS", nu),
        "unit_partial_begin": arr("OFF_UNIT_PARTIAL_BEGIN", nu),
        "split_units": arr("OFF_UNIT_LIST", h["N_SPLIT"]),
        "empty_units": buf[h["OFF_UNIT_LIST"] + h["N_SPLIT"]:
                           h["OFF_UNIT_LIST"] + h["N_SPLIT"] + h["N_EMPTY"]].tolist(),
        "cta_cost": buf[h["OFF_CTA_COST"]:h["OFF_CTA_COST"] + 2 * nc].view(np.float64).tolist(),
        "n_partials": h["N_PARTIALS"],
        "order": arr("OFF_WORK_ORDER", nw),
        "order_rec": [tuple(buf[h["OFF_ORDER_REC"] + 4 * i:h["OFF_ORDER_REC"] + 4 * i + 4].tolist())
                      for i in range(nw)],
    }
