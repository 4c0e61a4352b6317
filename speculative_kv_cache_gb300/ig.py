"""Python binding of libig.so: the C ABI of include/ig.h, same names, argument marshalling only.

Every function takes plain integers/floats for sizes and, for buffers, a torch tensor, a
NumPy array, a raw integer address, or None (NULL).  Nothing here computes: each call goes
straight to the library, and a non-zero status raises :class:`IGError`.  There is no fallback:
if libig.so is missing or cannot load, importing this module fails.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import numpy as np

try:  # torch provides the CUDA runtime that libig.so shares, and the tensors we pass
    import torch
except ImportError:  # pragma: no cover - torch is part of the environment
    torch = None

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libig.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "ig.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run `python -m speculative_kv_cache_gb300.build`")
_lib = C.CDLL(LIB_PATH)

IG_OK = 0
IG_ERR_INVALID = -1
IG_ERR_CUDA = -2
IG_ERR_OOM = -3
IG_ERR_NUMERIC = -4
IG_ERR_TIMEOUT = -5
IG_ERR_CAPACITY = -6
IG_SEL_THRESHOLD = 0
IG_SEL_HEAD_AVG = 1
IG_SEL_NORMALIZED = 2
IG_POOL_COUNTER = 0
IG_POOL_FIFO = 1
IG_POOL_LRU = 2
IG_POOL_NO_STORAGE = 1
IG_POOL_FP8 = 2
IG_POOL_INT4 = 4

_vp, _i, _f, _sz = C.c_void_p, C.c_int, C.c_float, C.c_size_t


class IGError(RuntimeError):
    def __init__(self, status: int, fn: str):
        self.status = status
        msg = _lib.ig_last_error().decode(errors="replace")
        super().__init__(f"{fn} failed with status {status}: {msg}")


def _sig(name, restype, *argtypes):
    f = getattr(_lib, name)
    f.restype = restype
    f.argtypes = list(argtypes)
    return f


_sig("ig_last_error", C.c_char_p)
_sig("ig_version", _i)
_sig("ig_check", _i, _vp)
_sig("ig_set_wait_limit", _i, _i)
_sig("ig_link_read", _i, _vp, _vp, _sz, _vp, _i)
_sig("ig_link_gather", _i, _vp, _vp, _sz, _i, _vp, _sz, _vp, _i)
_sig("ig_skew_weights", _i, _i, _i, _i, _f, _f, _vp, _i, _vp, _vp, _vp, _i, _vp, _vp, _vp, _vp,
     _vp, _vp, _i)
_sig("ig_skew_spectrum", _i, _i, _i, _i, _f, _vp, _i, _vp, _vp, _i)
_sig("ig_ratio_from_spectrum", _i, _i, _i, _vp, _f, C.POINTER(_i))
_sig("ig_speculate_workspace_bytes", _sz, _i, _i, _i, _i)
_sig("ig_speculate", _i, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _f, _vp, _vp, _vp, _sz)
_sig("ig_speculate_static", _i, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _f, _vp, _vp)
_sig("ig_speculate_rope_workspace_bytes", _sz, _i, _i, _i, _i, _i)
_sig("ig_speculate_rope", _i, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _f, _vp, _vp, _f,
     _vp, _vp, _vp, _sz)
_sig("ig_select_workspace_bytes", _sz, _i, _i)
_sig("ig_speculate_select_workspace_bytes", _sz, _i, _i, _i, _i, _i, _i)
_sig("ig_speculate_select", _i, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _f, _vp, _vp, _f, _f, _vp, _vp,
     _vp, _vp, _vp, _vp, _sz)
_sig("ig_select", _i, _vp, _i, _i, _i, _vp, _vp, _f, _i, _f, _vp, _vp, _vp, _vp, _sz)
_sig("ig_pool_create", _i, _i, _i, _i, _i, _i, C.POINTER(_vp))
_sig("ig_pool_create_ex", _i, _i, _i, _i, _i, _i, _i, _i, C.POINTER(_vp))
_sig("ig_pool_slot_tokens", _i, _vp, _i, _i, _vp)
_sig("ig_pool_kv8", _i, _vp, _i, C.POINTER(_vp), C.POINTER(_i), C.POINTER(_vp))
_sig("ig_pool_read_scales", _i, _vp, _i, _vp)
_sig("ig_pool_evictions", _i, _vp, _i, _i, C.POINTER(C.c_int64))
_sig("ig_append_kv_layers", _i, _vp, _vp, _i, _i, _i, _i, _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp)
_sig("ig_eviction_misses", _i, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp)
_sig("ig_prefill_workspace_bytes", _sz, _i, _i, _i, _i)
_sig("ig_prefill_layer", _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz)
_sig("ig_gemm_tn", _i, _vp, _i, _i, _i, _vp, _vp, _vp, _vp)
_sig("ig_prefill_layer_rope", _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
     _vp, _vp, _sz)
_sig("ig_attention_recall", _i, _vp, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _vp, _vp, _vp)
_sig("ig_captured_fraction", _i, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp)
_sig("ig_pool_destroy", _i, _vp)
_sig("ig_pool_kv", _i, _vp, _i, C.POINTER(_vp), C.POINTER(_vp))
_sig("ig_pool_write", _i, _vp, _vp, _i, _vp, _vp)
_sig("ig_pool_evict", _i, _vp, _i, _i, _vp, C.POINTER(C.c_int32), C.POINTER(C.c_int32))
_sig("ig_pool_counters", _i, _vp, _i, _i, _vp)
_sig("ig_gather_kv", _i, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _i)
_sig("ig_attend_workspace_bytes", _sz, _i, _i, _i, _i)
_sig("ig_sparse_attend", _i, _vp, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz)
_sig("ig_gather_attend_workspace_bytes", _sz, _i, _i, _i, _i)
_sig("ig_gather_attend", _i, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i)
_sig("ig_dense_attend", _i, _vp, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz)
_sig("ig_append_kv", _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp)


def header_functions() -> list[str]:
    """Names of the functions include/ig.h declares."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(ig_[a-z_0-9]+)\s*\(", txt)))


def _p(x):
    """Address of a buffer argument (tensor, ndarray, int, or None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if torch is not None and isinstance(x, torch.Tensor):
        if not x.is_contiguous():
            raise ValueError("tensor arguments must be contiguous")
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        if not x.flags["C_CONTIGUOUS"]:
            raise ValueError("array arguments must be C-contiguous")
        return x.ctypes.data
    raise TypeError(f"unsupported buffer argument {type(x)}")


def _s(stream):
    """A cudaStream_t from a torch stream, an int handle, or None (torch's current stream)."""
    if stream is None:
        if torch is not None and torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ok(st: int, fn: str):
    if st != IG_OK:
        raise IGError(st, fn)


def ig_version() -> int:
    return _lib.ig_version()


def ig_last_error() -> str:
    return _lib.ig_last_error().decode(errors="replace")


def ig_check(stream=None):
    _ok(_lib.ig_check(_s(stream)), "ig_check")


def ig_set_wait_limit(max_iters: int):
    _ok(_lib.ig_set_wait_limit(int(max_iters)), "ig_set_wait_limit")


def ig_link_read(stream, src, nbytes, sink, ctas=0):
    _ok(_lib.ig_link_read(_s(stream), _p(src), int(nbytes), _p(sink), int(ctas)), "ig_link_read")


def ig_link_gather(stream, src, rows, row_bytes, idx, n, dst, ctas=0):
    _ok(_lib.ig_link_gather(_s(stream), _p(src), int(rows), int(row_bytes), _p(idx), int(n), _p(dst), int(ctas)),
        "ig_link_gather")


def ig_skew_weights(D, H, d, ratio, rope_theta, Xs, Ns, Wq, Wk, Kp, Nk, A, Wq_skew, Wk_skew,
                    Kp_skew, cols, threads=0) -> int:
    k = C.c_int(0)
    _ok(_lib.ig_skew_weights(D, H, d, ratio, rope_theta, _p(Xs), Ns, _p(Wq), _p(Wk), _p(Kp), Nk,
                             _p(A), _p(Wq_skew), _p(Wk_skew), _p(Kp_skew), _p(cols), C.byref(k),
                             threads), "ig_skew_weights")
    return k.value


def ig_skew_spectrum(D, H, d, rope_theta, Xs, Ns, Wq, sigma, threads=0):
    _ok(_lib.ig_skew_spectrum(D, H, d, rope_theta, _p(Xs), Ns, _p(Wq), _p(sigma), threads), "ig_skew_spectrum")


def ig_ratio_from_spectrum(H, d, sigma, energy) -> int:
    k = C.c_int(0)
    _ok(_lib.ig_ratio_from_spectrum(H, d, _p(sigma), energy, C.byref(k)), "ig_ratio_from_spectrum")
    return k.value


def ig_speculate_workspace_bytes(B, D, H, k) -> int:
    return _lib.ig_speculate_workspace_bytes(B, D, H, k)


def ig_speculate(stream, B, D, H, k, Lcap, x, Wq_part, Kpart, L_valid, score_scale, scores,
                 q_part, workspace, workspace_bytes):
    _ok(_lib.ig_speculate(_s(stream), B, D, H, k, Lcap, _p(x), _p(Wq_part), _p(Kpart), _p(L_valid),
                          score_scale, _p(scores), _p(q_part), _p(workspace), workspace_bytes),
        "ig_speculate")


def ig_speculate_static(stream, B, D, H, k, Lcap, x, Wq_part, Kpart, L_valid, score_scale, scores,
                        q_part):
    """ig_speculate with the library's own static scratch: no workspace, nothing allocated."""
    _ok(_lib.ig_speculate_static(_s(stream), B, D, H, k, Lcap, _p(x), _p(Wq_part), _p(Kpart),
                                 _p(L_valid), score_scale, _p(scores), _p(q_part)),
        "ig_speculate_static")


def ig_speculate_rope_workspace_bytes(B, D, H, d, k) -> int:
    return _lib.ig_speculate_rope_workspace_bytes(B, D, H, d, k)


def ig_speculate_rope(stream, B, D, H, d, k, Lcap, x, Wq, A_cols, positions, rope_theta, Kpart,
                      L_valid, score_scale, scores, q_part, workspace, workspace_bytes):
    _ok(_lib.ig_speculate_rope(_s(stream), B, D, H, d, k, Lcap, _p(x), _p(Wq), _p(A_cols),
                               _p(positions), rope_theta, _p(Kpart), _p(L_valid), score_scale,
                               _p(scores), _p(q_part), _p(workspace), workspace_bytes),
        "ig_speculate_rope")


def ig_select_workspace_bytes(B, H) -> int:
    return _lib.ig_select_workspace_bytes(B, H)


def ig_select(stream, B, H, Lcap, scores, L_valid, alpha, policy, cap_frac, idx, cnt, used,
              workspace=None, workspace_bytes=0):
    _ok(_lib.ig_select(_s(stream), B, H, Lcap, _p(scores), _p(L_valid), alpha, policy, cap_frac,
                       _p(idx), _p(cnt), _p(used), _p(workspace), workspace_bytes), "ig_select")


def ig_speculate_select_workspace_bytes(B, D, H, d, k, rope) -> int:
    return _lib.ig_speculate_select_workspace_bytes(B, D, H, d, k, int(bool(rope)))


def ig_speculate_select(stream, B, D, H, d, k, Lcap, x, Wq, A_cols, positions, rope_theta, Kpart, L_valid,
                        score_scale, alpha, idx, cnt, used, scores, q_part, workspace, workspace_bytes):
    _ok(_lib.ig_speculate_select(_s(stream), B, D, H, d, k, Lcap, _p(x), _p(Wq), _p(A_cols), _p(positions),
                                 rope_theta, _p(Kpart), _p(L_valid), score_scale, alpha, _p(idx), _p(cnt),
                                 _p(used), _p(scores), _p(q_part), _p(workspace), workspace_bytes),
        "ig_speculate_select")


def ig_pool_create(layers, B, H, d, cap) -> int:
    h = _vp()
    _ok(_lib.ig_pool_create(layers, B, H, d, cap, C.byref(h)), "ig_pool_create")
    return h.value


def ig_pool_create_ex(layers, B, H, d, cap, policy=IG_POOL_COUNTER, flags=0) -> int:
    h = _vp()
    _ok(_lib.ig_pool_create_ex(layers, B, H, d, cap, policy, flags, C.byref(h)), "ig_pool_create_ex")
    return h.value


def ig_pool_destroy(pool):
    _ok(_lib.ig_pool_destroy(pool), "ig_pool_destroy")


def ig_pool_kv(pool, layer):
    """Host addresses (also valid on the device) of one layer's K and V arrays."""
    k, v = _vp(), _vp()
    _ok(_lib.ig_pool_kv(pool, layer, C.byref(k), C.byref(v)), "ig_pool_kv")
    return k.value, v.value


def ig_pool_write(pool, stream, layer, K, V):
    _ok(_lib.ig_pool_write(pool, _s(stream), layer, _p(K), _p(V)), "ig_pool_write")


def ig_pool_evict(pool, layer, b, used):
    slot, filled = C.c_int32(0), C.c_int32(0)
    _ok(_lib.ig_pool_evict(pool, layer, b, _p(used), C.byref(slot), C.byref(filled)), "ig_pool_evict")
    return slot.value, filled.value


def ig_pool_counters(pool, layer, b, out):
    _ok(_lib.ig_pool_counters(pool, layer, b, _p(out)), "ig_pool_counters")


def ig_pool_kv8(pool, layer):
    """Quantized pools: host address (also valid on the device) of one layer's code records, the
    record size, and the device address of that layer's scales [B][H][cap][2]."""
    r, n, sp = _vp(), _i(0), _vp()
    _ok(_lib.ig_pool_kv8(pool, layer, C.byref(r), C.byref(n), C.byref(sp)), "ig_pool_kv8")
    return r.value, n.value, sp.value


def ig_pool_read_scales(pool, layer, out):
    _ok(_lib.ig_pool_read_scales(pool, layer, _p(out)), "ig_pool_read_scales")


def _pool_layer_view_q(pool, layer, B, H, cap, cb):
    r, rec, _ = ig_pool_kv8(pool, layer)
    raw = np.ctypeslib.as_array(C.cast(r, C.POINTER(C.c_uint8)), shape=(B * H * cap * rec,)).reshape(B, H, cap, rec)
    sc = np.zeros((B, H, cap, 2), dtype=np.float32)
    ig_pool_read_scales(pool, layer, sc)
    return raw[..., :cb], raw[..., cb:2 * cb], sc[..., 0], sc[..., 1]


def pool_layer_view_fp8(pool, layer, B, H, cap, d):
    """One layer of an fp8 pool: codes [B, H, cap, d] uint8 (K, V; views into the pinned
    records) and scales [B, H, cap] float32 (K, V; a copy of the device-resident scales)."""
    return _pool_layer_view_q(pool, layer, B, H, cap, d)


def pool_layer_view_int4(pool, layer, B, H, cap, d):
    """One layer of an int4 pool: packed codes [B, H, cap, d/2] uint8 (K, V; two codes per byte,
    element 2j in the low nibble; views into the pinned records) and scales [B, H, cap] float32
    (K, V; a copy of the device-resident scales)."""
    return _pool_layer_view_q(pool, layer, B, H, cap, d // 2)


def ig_pool_slot_tokens(pool, layer, b, out):
    _ok(_lib.ig_pool_slot_tokens(pool, layer, b, _p(out)), "ig_pool_slot_tokens")


def ig_pool_evictions(pool, layer, b) -> int:
    n = C.c_int64()
    _ok(_lib.ig_pool_evictions(pool, layer, b, C.byref(n)), "ig_pool_evictions")
    return n.value


def ig_eviction_misses(stream, B, H, Lcap, scores, idx, cnt, resident, miss_cnt, miss_mass):
    _ok(_lib.ig_eviction_misses(_s(stream), B, H, Lcap, _p(scores), _p(idx), _p(cnt), _p(resident),
                                _p(miss_cnt), _p(miss_mass)), "ig_eviction_misses")


def ig_prefill_workspace_bytes(B, N, H, d):
    return _lib.ig_prefill_workspace_bytes(B, N, H, d)


def ig_prefill_layer(stream, pool, layer, B, N, D, H, d, k, Lcap, X, Wq_t, Wk_t, Wv_t, cols, Wq_part_t, Kpart,
                     workspace, workspace_bytes):
    _ok(_lib.ig_prefill_layer(_s(stream), pool, layer, B, N, D, H, d, k, Lcap, _p(X), _p(Wq_t), _p(Wk_t), _p(Wv_t),
                              _p(cols), _p(Wq_part_t), _p(Kpart), _p(workspace), workspace_bytes),
        "ig_prefill_layer")


def ig_prefill_layer_rope(stream, pool, layer, B, N, D, H, d, k, Lcap, rope_theta, X, Wq_t, Wk_t, Wv_t, A, cols,
                          A_cols, Kpart, workspace, workspace_bytes):
    _ok(_lib.ig_prefill_layer_rope(_s(stream), pool, layer, B, N, D, H, d, k, Lcap, rope_theta, _p(X), _p(Wq_t),
                                   _p(Wk_t), _p(Wv_t), _p(A), _p(cols), _p(A_cols), _p(Kpart), _p(workspace),
                                   workspace_bytes), "ig_prefill_layer_rope")


def ig_gemm_tn(stream, M, N, K, A, Bt, C, colpart=None):
    _ok(_lib.ig_gemm_tn(_s(stream), M, N, K, _p(A), _p(Bt), _p(C), _p(colpart)), "ig_gemm_tn")


def ig_attention_recall(stream, B, H, d, Lcap, scale, q, K, L_valid, idx, cnt, recall, weight):
    _ok(_lib.ig_attention_recall(_s(stream), B, H, d, Lcap, scale, _p(q), _p(K), _p(L_valid), _p(idx), _p(cnt),
                                 _p(recall), _p(weight)), "ig_attention_recall")


def ig_captured_fraction(stream, B, H, d, k, Lcap, q, K, L_valid, cols, frac):
    _ok(_lib.ig_captured_fraction(_s(stream), B, H, d, k, Lcap, _p(q), _p(K), _p(L_valid), _p(cols), _p(frac)),
        "ig_captured_fraction")


def ig_gather_kv(stream, pool, layer, B, H, d, Lcap, idx, cnt, Kg, Vg, max_ctas=0):
    _ok(_lib.ig_gather_kv(_s(stream), pool, layer, B, H, d, Lcap, _p(idx), _p(cnt), _p(Kg), _p(Vg),
                          max_ctas), "ig_gather_kv")


def ig_attend_workspace_bytes(B, H, d, Lcap) -> int:
    return _lib.ig_attend_workspace_bytes(B, H, d, Lcap)


def ig_sparse_attend(stream, B, H, d, Lcap, scale, q, Kg, Vg, cnt, k_new, v_new, out, workspace,
                     workspace_bytes):
    _ok(_lib.ig_sparse_attend(_s(stream), B, H, d, Lcap, scale, _p(q), _p(Kg), _p(Vg), _p(cnt),
                              _p(k_new), _p(v_new), _p(out), _p(workspace), workspace_bytes),
        "ig_sparse_attend")


def ig_gather_attend_workspace_bytes(B, H, d, Lcap):
    return _lib.ig_gather_attend_workspace_bytes(B, H, d, Lcap)


def ig_gather_attend(stream, pool, layer, B, H, d, Lcap, scale, q, idx, cnt, k_new, v_new, out,
                     workspace, workspace_bytes, max_ctas=0):
    _ok(_lib.ig_gather_attend(_s(stream), pool, layer, B, H, d, Lcap, scale, _p(q), _p(idx), _p(cnt),
                              _p(k_new), _p(v_new), _p(out), _p(workspace), workspace_bytes, max_ctas),
        "ig_gather_attend")


def ig_dense_attend(stream, B, H, d, Lcap, scale, q, K, V, L_valid, k_new, v_new, out, workspace,
                    workspace_bytes):
    _ok(_lib.ig_dense_attend(_s(stream), B, H, d, Lcap, scale, _p(q), _p(K), _p(V), _p(L_valid),
                             _p(k_new), _p(v_new), _p(out), _p(workspace), workspace_bytes),
        "ig_dense_attend")


def ig_append_kv(stream, pool, layer, B, H, d, k, Lcap, slot, cols, k_new, v_new, Kpart, Kdense=None,
                 Vdense=None):
    _ok(_lib.ig_append_kv(_s(stream), pool, layer, B, H, d, k, Lcap, _p(slot), _p(cols), _p(k_new),
                          _p(v_new), _p(Kpart), _p(Kdense), _p(Vdense)), "ig_append_kv")


def ig_append_kv_layers(stream, pool, layers, B, H, d, ks, Lcap, slot, cols, k_new, v_new, Kpart, Kdense=None,
                        Vdense=None):
    """ks: list of ints; cols, Kpart: lists of device tensors (or None entries)."""
    ks_a = (C.c_int * layers)(*[int(x) for x in ks])
    cols_a = _ptr_array(cols)
    kp_a = _ptr_array(Kpart) if Kpart is not None else None
    _ok(_lib.ig_append_kv_layers(_s(stream), pool, layers, B, H, d, C.cast(ks_a, _vp), Lcap, _p(slot),
                                 C.cast(cols_a, _vp), _p(k_new), _p(v_new),
                                 C.cast(kp_a, _vp) if kp_a is not None else None, _p(Kdense), _p(Vdense)),
        "ig_append_kv_layers")


def pool_layer_view(pool, layer, B, H, cap, d):
    """NumPy views (fp16) of one layer's K and V in the pinned pool: [B, H, cap, d] each."""
    kp, vp = ig_pool_kv(pool, layer)
    n = B * H * cap * d
    K = np.ctypeslib.as_array(C.cast(kp, C.POINTER(C.c_uint16)), shape=(n,)).view(np.float16)
    V = np.ctypeslib.as_array(C.cast(vp, C.POINTER(C.c_uint16)), shape=(n,)).view(np.float16)
    return K.reshape(B, H, cap, d), V.reshape(B, H, cap, d)


# ---------------------------------------------------------------------------------------
# Decoder (one step over every layer) and the batched pool manager
# ---------------------------------------------------------------------------------------
class DecoderConfig(C.Structure):
    _fields_ = [("layers", _i), ("B", _i), ("H", _i), ("d", _i), ("D", _i), ("k", _i), ("Lcap", _i),
                ("policy", _i), ("alpha", _f), ("cap_frac", _f), ("score_scale", _f),
                ("rope_theta", _f), ("gather_ctas", _i), ("stage_timing", _i), ("fused_select", _i),
                ("fused_fetch", _i), ("batched_append", _i), ("append_on_fetch", _i),
                ("keep_indices", _i)]


class DecoderBuffers(C.Structure):
    _fields_ = [("Wq_part", C.POINTER(_vp)), ("Wq", C.POINTER(_vp)), ("A_cols", C.POINTER(_vp)),
                ("Kpart", C.POINTER(_vp)), ("cols", C.POINTER(_vp)), ("K0", _vp), ("V0", _vp),
                ("scores", _vp), ("idx", _vp), ("cnt", _vp), ("used", _vp), ("Kg", _vp), ("Vg", _vp),
                ("workspace", _vp), ("workspace_bytes", _sz), ("ks", C.POINTER(_i))]


class StepIO(C.Structure):
    _fields_ = [("x", _vp), ("q", _vp), ("k_new", _vp), ("v_new", _vp), ("L_valid", _vp),
                ("positions", _vp), ("slot", _vp), ("out", _vp)]


_sig("ig_decoder_workspace_bytes", _sz, C.POINTER(DecoderConfig))
_sig("ig_decoder_create", _i, C.POINTER(DecoderConfig), C.POINTER(DecoderBuffers), _vp, C.POINTER(_vp))
_sig("ig_decoder_destroy", _i, _vp)
_sig("ig_decode_step", _i, _vp, C.POINTER(StepIO), _vp, _vp)
_sig("ig_decoder_stage_ms", _i, _vp, _i, C.POINTER(_f), C.POINTER(_i))
_sig("ig_decoder_timeline", _i, _vp, _i, C.POINTER(_f))
_sig("ig_pool_update", _i, _vp, _i, _i, _vp)
_sig("ig_pool_prefill", _i, _vp, _i, _vp)
_sig("ig_pool_step", _i, _vp, _vp, _i, _vp)
_sig("ig_pool_full", _i, _vp, C.POINTER(_i))
_sig("ig_launch_count", C.c_uint64)
_sig("ig_sm_split_create", _i, _i, _i, C.POINTER(_vp), C.POINTER(_vp), C.POINTER(_vp), C.POINTER(_i), C.POINTER(_i))
_sig("ig_sm_split_destroy", _i, _vp)
_sig("ig_decoder_graph_capture", _i, _vp, C.POINTER(StepIO), _vp, _vp)
_sig("ig_decoder_graph_launch", _i, _vp, _vp)


def _ptr_array(items):
    arr = (_vp * len(items))(*[_p(t) for t in items])
    return arr


def ig_decoder_workspace_bytes(cfg: DecoderConfig) -> int:
    return _lib.ig_decoder_workspace_bytes(C.byref(cfg))


def ig_decoder_create(cfg: DecoderConfig, bufs: DecoderBuffers, pool) -> int:
    h = _vp()
    _ok(_lib.ig_decoder_create(C.byref(cfg), C.byref(bufs), pool, C.byref(h)), "ig_decoder_create")
    return h.value


def ig_decoder_destroy(dec):
    _ok(_lib.ig_decoder_destroy(dec), "ig_decoder_destroy")


def ig_decode_step(dec, io: StepIO, stream, side_stream):
    _ok(_lib.ig_decode_step(dec, C.byref(io), _s(stream), _s(side_stream)), "ig_decode_step")


def ig_decoder_graph_capture(dec, io: StepIO, stream, side_stream):
    _ok(_lib.ig_decoder_graph_capture(dec, C.byref(io), _s(stream), _s(side_stream)), "ig_decoder_graph_capture")


def ig_decoder_graph_launch(dec, stream):
    _ok(_lib.ig_decoder_graph_launch(dec, _s(stream)), "ig_decoder_graph_launch")


def ig_decoder_stage_ms(dec, steps_back=0):
    ms = (_f * 4)()
    cnt = (_i * 4)()
    _ok(_lib.ig_decoder_stage_ms(dec, steps_back, ms, cnt), "ig_decoder_stage_ms")
    return list(ms), list(cnt)


def ig_decoder_timeline(dec, layers, steps_back=0):
    """[layers, 6] float32: fetch start/end, speculate+select start/end, attend+append
    start/end (ms from the step's first timed stage; NaN where a layer has no such stage)."""
    t = np.zeros((layers, 6), dtype=np.float32)
    _ok(_lib.ig_decoder_timeline(dec, steps_back, t.ctypes.data_as(C.POINTER(_f))), "ig_decoder_timeline")
    return t


def ig_pool_update(pool, layer, b, used):
    _ok(_lib.ig_pool_update(pool, layer, b, _p(used)), "ig_pool_update")


def ig_pool_prefill(pool, n_tokens, slots_out=None):
    _ok(_lib.ig_pool_prefill(pool, n_tokens, _p(slots_out)), "ig_pool_prefill")


def ig_pool_step(pool, used, Lcap, slots_out):
    _ok(_lib.ig_pool_step(pool, _p(used), Lcap, _p(slots_out)), "ig_pool_step")


def ig_pool_full(pool) -> bool:
    f = _i(0)
    _ok(_lib.ig_pool_full(pool, C.byref(f)), "ig_pool_full")
    return bool(f.value)


def ig_launch_count() -> int:
    return _lib.ig_launch_count()


def ig_sm_split_create(device: int, fetch_sms: int):
    """(split handle, compute stream handle, fetch stream handle, compute SMs, fetch SMs)."""
    h, cs, fs = _vp(), _vp(), _vp()
    nc, nf = _i(), _i()
    _ok(_lib.ig_sm_split_create(device, fetch_sms, C.byref(h), C.byref(cs), C.byref(fs), C.byref(nc), C.byref(nf)),
        "ig_sm_split_create")
    return h.value, cs.value, fs.value, nc.value, nf.value


def ig_sm_split_destroy(split):
    _ok(_lib.ig_sm_split_destroy(split), "ig_sm_split_destroy")
