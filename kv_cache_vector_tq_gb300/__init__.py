"""TurboQuant hot path on GB300 (sm_103a): Python binding of the libtq C ABI.

The functions here marshal arguments (torch tensors -> device pointers, numpy
arrays -> host pointers) and call libtq.so; every step of the path runs in the
library's kernels.  The library is built in-tree by ``build.build()``; when it
is missing, ``lib()`` raises instead of falling back to anything else.
"""

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libtq.so")

TQ_OK, TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_CUDA, TQ_ERR_ALLOC, TQ_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
TQ_MSE, TQ_PROD, TQ_MIXED = 0, 1, 2
TQ_ROT_DENSE, TQ_ROT_HADAMARD = 0, 1
TQ_DENS_BETA, TQ_DENS_GAUSS = 0, 1
TQ_F32, TQ_F16 = 0, 1
TQ_LAYOUT_TOKEN, TQ_LAYOUT_PAIR = 0, 1

# every entry point of include/tq.h
EXPORTS = (
    "tq_version", "tq_status_string", "tq_last_cuda_error", "tq_codebook_build",
    "tq_rotation_haar", "tq_ctx_create", "tq_ctx_destroy", "tq_codes_layout", "tq_encode",
    "tq_scores_workspace_size", "tq_scores", "tq_decode_workspace_size",
    "tq_decode_attention", "tq_decode_step", "tq_decode_attention_noalloc", "tq_unpack_indices", "tq_status_poll",
    "tq_ctx_set_wait_limit",
)


class TqError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = _LIB.tq_status_string(status).decode() if _LIB else str(status)
        if status == TQ_ERR_CUDA and _LIB:
            msg += f" (cudaError {_LIB.tq_last_cuda_error()})"
        super().__init__(f"{fn}: {msg}")


class Codebook(ctypes.Structure):
    _fields_ = [
        ("d", ctypes.c_int), ("b", ctypes.c_int), ("density", ctypes.c_int),
        ("grid", ctypes.c_int), ("iters", ctypes.c_int),
        ("centroid", ctypes.c_double * 16), ("threshold", ctypes.c_double * 15),
        ("distortion", ctypes.c_double),
    ]


class Codes(ctypes.Structure):
    _fields_ = [
        ("d_codes", ctypes.c_void_p), ("d_norm", ctypes.c_void_p),
        ("d_qjl", ctypes.c_void_p), ("d_rnorm", ctypes.c_void_p),
        ("n", ctypes.c_int64), ("d", ctypes.c_int), ("b_mse", ctypes.c_int),
        ("mode", ctypes.c_int), ("layout", ctypes.c_int),
        ("words_per_vec", ctypes.c_int), ("qjl_words_per_vec", ctypes.c_int),
    ]


_LIB = None
_vp, _i, _i64, _sz, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float


def lib():
    """Load libtq.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libtq.so is not built ({LIB_PATH}); run kv_cache_vector_tq_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    sig = {
        "tq_version": ([], ctypes.c_char_p),
        "tq_status_string": ([_i], ctypes.c_char_p),
        "tq_last_cuda_error": ([], _i),
        "tq_codebook_build": ([_i, _i, _i, _i, _i, P(Codebook)], _i),
        "tq_rotation_haar": ([_i, _vp, _vp], _i),
        "tq_ctx_create": ([_i, _i, _i, _i, _vp, _vp, P(Codebook), P(_vp)], _i),
        "tq_ctx_destroy": ([_vp], _i),
        "tq_codes_layout": ([_vp, _i, _i64, P(Codes), P(_sz), P(_sz), P(_sz), P(_sz)], _i),
        "tq_encode": ([_vp, _vp, _i, _i64, P(Codes), _i64, _i64, _i64, _vp], _i),
        "tq_scores_workspace_size": ([_vp, _i, P(_sz)], _i),
        "tq_scores": ([_vp, _vp, _i, P(Codes), _i64, _i64, _vp, _vp, _sz, _vp], _i),
        "tq_decode_workspace_size": ([_vp, _i, _i, _i, _i64, P(_sz)], _i),
        "tq_decode_attention": ([_vp, _vp, _vp, _i, P(Codes), P(Codes), _i, _i, _i, _i64, _i64,
                                 _f, _vp, _vp, _sz, _vp], _i),
        "tq_decode_step": ([_vp, _vp, _vp, _i, _vp, _vp, _i, P(Codes), P(Codes), _i, _i, _i, _i64,
                            _i64, _f, _vp, _vp, _sz, _vp], _i),
        "tq_decode_attention_noalloc": ([_vp, _vp, _vp, _i, P(Codes), P(Codes), _i, _i, _i, _i64,
                                         _i64, _f, _vp, _vp], _i),
        "tq_unpack_indices": ([P(Codes), _i64, _i64, _vp, _vp], _i),
        "tq_status_poll": ([_vp, _vp], _i),
        "tq_ctx_set_wait_limit": ([_vp, ctypes.c_uint32], _i),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _LIB = L
    return L


def _check(fn, st):
    if st != TQ_OK:
        raise TqError(fn, st)


def _ptr(a):
    """Host pointer of a contiguous numpy array."""
    return a.ctypes.data_as(ctypes.c_void_p)


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


# ---------------------------------------------------------------- host calls
def tq_version():
    return lib().tq_version().decode()


def tq_codebook_build(d, b, density=TQ_DENS_BETA, grid=0, iters=0):
    cb = Codebook()
    _check("tq_codebook_build", lib().tq_codebook_build(d, b, density, grid, iters, ctypes.byref(cb)))
    return cb


def tq_rotation_haar(G):
    import numpy as np
    G = np.ascontiguousarray(G, dtype=np.float64)
    d = G.shape[0]
    Pi = np.empty((d, d), dtype=np.float64)
    _check("tq_rotation_haar", lib().tq_rotation_haar(d, _ptr(G), _ptr(Pi)))
    return Pi


class Context:
    """Owns a tq_ctx (device tables for one (d, b, mode, rotation)).  TQ_MIXED
    (b + 1/2 bits per coordinate) passes the b-bit and (b+1)-bit codebooks."""

    def __init__(self, d, b, mode, rot_kind, rot, S=None, codebook=None):
        import numpy as np
        rot = np.ascontiguousarray(rot, dtype=np.float64)
        S = None if S is None else np.ascontiguousarray(S, dtype=np.float64)
        self.d, self.b, self.mode, self.rot_kind = d, b, mode, rot_kind
        self.b_mse = b - 1 if mode == TQ_PROD else b
        if mode == TQ_MIXED:
            pair = (Codebook * 2)()
            pair[0] = tq_codebook_build(d, b) if codebook is None else codebook[0]
            pair[1] = tq_codebook_build(d, b + 1) if codebook is None else codebook[1]
            self.codebook = pair
        else:
            self.codebook = codebook if codebook is not None else tq_codebook_build(d, self.b_mse)
        h = ctypes.c_void_p()
        cbp = (ctypes.cast(self.codebook, ctypes.POINTER(Codebook)) if mode == TQ_MIXED
               else ctypes.byref(self.codebook))
        _check("tq_ctx_create", lib().tq_ctx_create(
            d, b, mode, rot_kind, _ptr(rot), _ptr(S) if S is not None else None, cbp, ctypes.byref(h)))
        self.handle = h

    def close(self):
        if self.handle:
            _check("tq_ctx_destroy", lib().tq_ctx_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_wait_limit(self, polls):
        """Bound of the context's pipeline waits (tq_ctx_set_wait_limit)."""
        _check("tq_ctx_set_wait_limit", lib().tq_ctx_set_wait_limit(self.handle, int(polls)))

    def poll(self, stream=None):
        st = lib().tq_status_poll(self.handle, _stream(stream))
        return st


class CodeSet:
    """Packed codes of n vectors in device memory (torch tensors)."""

    def __init__(self, ctx, n, layout=TQ_LAYOUT_TOKEN, device="cuda"):
        import torch
        desc = Codes()
        sizes = [ctypes.c_size_t() for _ in range(4)]
        _check("tq_codes_layout", lib().tq_codes_layout(ctx.handle, layout, n, ctypes.byref(desc),
                                                        *[ctypes.byref(s) for s in sizes]))
        cb, nb, qb, rb = (s.value for s in sizes)
        self.codes = torch.zeros(max(cb // 4, 4), dtype=torch.int32, device=device)
        self.norm = torch.zeros(max(nb // 4, 4), dtype=torch.float32, device=device)
        self.qjl = torch.zeros(max(qb // 4, 4), dtype=torch.int32, device=device) if qb else None
        self.rnorm = torch.zeros(max(rb // 4, 4), dtype=torch.float32, device=device) if rb else None
        desc.d_codes = self.codes.data_ptr()
        desc.d_norm = self.norm.data_ptr()
        desc.d_qjl = self.qjl.data_ptr() if self.qjl is not None else None
        desc.d_rnorm = self.rnorm.data_ptr() if self.rnorm is not None else None
        self.desc = desc
        self.n, self.layout, self.ctx = n, layout, ctx

    @property
    def words_per_vec(self):
        return self.desc.words_per_vec


# ---------------------------------------------------------------- device calls
def tq_encode(ctx, x, codes, offset=0, group_rows=None, group_stride=0, stream=None):
    import torch
    assert x.is_cuda and x.is_contiguous()
    dt = {torch.float32: TQ_F32, torch.float16: TQ_F16}[x.dtype]
    N = x.shape[0] if x.dim() == 2 else x.numel() // ctx.d
    gr = N if group_rows is None else group_rows
    _check("tq_encode", lib().tq_encode(ctx.handle, ctypes.c_void_p(x.data_ptr()), dt, N,
                                        ctypes.byref(codes.desc), offset, max(gr, 1), group_stride,
                                        _stream(stream)))


def tq_scores_workspace_size(ctx, M):
    n = ctypes.c_size_t()
    _check("tq_scores_workspace_size", lib().tq_scores_workspace_size(ctx.handle, M, ctypes.byref(n)))
    return n.value


def tq_scores(ctx, q, keys, out, ws, first=0, N=None, stream=None):
    N = keys.n - first if N is None else N
    M = q.shape[0]
    _check("tq_scores", lib().tq_scores(ctx.handle, ctypes.c_void_p(q.data_ptr()), M,
                                        ctypes.byref(keys.desc), first, N,
                                        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                                        ws.numel() * ws.element_size(), _stream(stream)))


def tq_decode_workspace_size(kctx, B, Hq, Hkv, seq):
    n = ctypes.c_size_t()
    _check("tq_decode_workspace_size",
           lib().tq_decode_workspace_size(kctx.handle, B, Hq, Hkv, seq, ctypes.byref(n)))
    return n.value


def tq_decode_attention(kctx, vctx, q, K, V, B, Hq, Hkv, seq, cap, scale, out, ws, stream=None):
    import torch
    dt = {torch.float32: TQ_F32, torch.float16: TQ_F16}[q.dtype]
    _check("tq_decode_attention", lib().tq_decode_attention(
        kctx.handle, vctx.handle, ctypes.c_void_p(q.data_ptr()), dt, ctypes.byref(K.desc),
        ctypes.byref(V.desc), B, Hq, Hkv, seq, cap, float(scale), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(), _stream(stream)))


def tq_decode_step(kctx, vctx, q, k_new, v_new, K, V, B, Hq, Hkv, seq, cap, scale, out, ws, stream=None):
    """Append k_new/v_new ([B, Hkv, d]) at position seq-1, then attend over seq tokens."""
    import torch
    dts = {torch.float32: TQ_F32, torch.float16: TQ_F16}
    assert k_new.dtype == v_new.dtype
    _check("tq_decode_step", lib().tq_decode_step(
        kctx.handle, vctx.handle, ctypes.c_void_p(q.data_ptr()), dts[q.dtype],
        ctypes.c_void_p(k_new.data_ptr()), ctypes.c_void_p(v_new.data_ptr()), dts[k_new.dtype],
        ctypes.byref(K.desc), ctypes.byref(V.desc), B, Hq, Hkv, seq, cap, float(scale),
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(),
        _stream(stream)))


def tq_decode_attention_noalloc(kctx, vctx, q, K, V, B, Hq, Hkv, seq, cap, scale, out, stream=None):
    """tq_decode_attention without a workspace (scratch built into the library)."""
    import torch
    dt = {torch.float32: TQ_F32, torch.float16: TQ_F16}[q.dtype]
    _check("tq_decode_attention_noalloc", lib().tq_decode_attention_noalloc(
        kctx.handle, vctx.handle, ctypes.c_void_p(q.data_ptr()), dt, ctypes.byref(K.desc),
        ctypes.byref(V.desc), B, Hq, Hkv, seq, cap, float(scale), ctypes.c_void_p(out.data_ptr()),
        _stream(stream)))


def tq_unpack_indices(codes, first=0, count=None, with_bits=False):
    import numpy as np
    count = codes.n - first if count is None else count
    idx = np.zeros((count, codes.desc.d), dtype=np.uint8)
    bits = np.zeros((count, codes.desc.d), dtype=np.uint8) if with_bits else None
    _check("tq_unpack_indices", lib().tq_unpack_indices(ctypes.byref(codes.desc), first, count,
                                                        _ptr(idx), _ptr(bits) if with_bits else None))
    return (idx, bits) if with_bits else idx
