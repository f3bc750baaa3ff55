"""Exact attention for GB300 (sm_103a): Python binding of the C ABI in
include/fa.h.

This module only marshals arguments: every step of the forward and backward
runs in the CUDA library libfa_gb300.so, built in-tree by
`__graft_entry__.build()`. There is no fallback: if the library is missing or
the device is not sm_103, the calls raise.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")

FA_OK = 0
_STATUS_NAMES = {
    0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_ARCH",
    4: "FA_ERR_CUDA", 5: "FA_ERR_TIMEOUT", 6: "FA_ERR_WORKSPACE", 7: "FA_ERR_DEVICE",
}

# Every symbol include/fa.h declares, with its ctypes signature.
_VP, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_LL = ctypes.c_longlong
SIGNATURES = {
    "fa_fwd": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_fwd_f32": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_fwd_kv": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_fwd_pair": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_bwd_kv": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ,
                       _I, _I, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_fwd_blocksparse": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _LL, _LL, _I, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_bwd_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "fa_bwd": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ,
                    _I, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_bwd_deterministic": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ,
                                  _I, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_bwd_blocksparse_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "fa_bwd_blocksparse": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _LL, _LL,
                                _I, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_bwd_preprocess": (_I, [_VP, _VP, _VP, _VP, _SZ, _I, _I, _I, _I, _I, _VP]),
    "fa_bwd_dkdv": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _I, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_bwd_dq": (_I, [_VP, _VP, _SZ, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_bwd_noalloc": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_fp8_row_scales": (_SZ, [_I]),
    "fa_fp8_vt_keys": (_SZ, [_I]),
    "fa_fp8_quantize_rows": (_I, [_VP, _VP, _VP, _I, _I, _I, _VP]),
    "fa_fp8_quantize_v": (_I, [_VP, _VP, _VP, _I, _I, _I, _VP]),
    "fa_fwd_fp8": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_fwd_fp8_kv": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _F, _VP]),
    "fa_ex2_throughput": (_I, [ctypes.POINTER(ctypes.c_double), _VP]),
    "fa_sm_clock_mhz": (_I, [ctypes.POINTER(ctypes.c_double), _VP]),
    "fa_device_status": (_I, [_VP]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_version": (_I, []),
}

_lib = None


class FAError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        msg = _lib.fa_status_string(code).decode() if _lib is not None else ""
        super().__init__(f"{fn} returned {_STATUS_NAMES.get(code, code)}: {msg}")


def load(path=None):
    """Load the compiled library (once) and declare its signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} (run __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(fn, code):
    if code != FA_OK:
        raise FAError(fn, code)


def _stream(t):
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _shape(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be 4-D: [B, H, N, d]")
    B, Hq, N, d = q.shape
    return B, Hq, k.shape[1], N, d


def _require(device, *specs):
    """Refuse, before any launch, a tensor the kernels would read or write past
    its end. specs: (tensor, name, dtype, shape). Every dtype and shape is
    checked before any placement (contiguous, CUDA, on the device of q), so
    the shape rules hold for CPU tensors too."""
    for t, name, dtype, shape in specs:
        if t.dtype != dtype or tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name}: expected {dtype} of shape {tuple(shape)}, "
                             f"got {t.dtype} of shape {tuple(t.shape)}")
    for t, name, _, _ in specs:
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not t.is_cuda or t.device != device:
            raise ValueError(f"{name} must be a CUDA tensor on {device}")


def _mask_args(block_mask, B, Hq, N, device):
    """Pointer and byte strides of a block mask tensor: uint8 or bool on the
    device, shape [B or 1, Hq or 1, T, T] with T = ceil(N / 128), the last two
    dimensions dense (a size-1 batch or head dimension broadcasts)."""
    import torch
    T = (N + 127) // 128
    if block_mask.dtype not in (torch.uint8, torch.bool) or block_mask.device != device:
        raise ValueError("block_mask must be a uint8 or bool tensor on the device of q")
    if block_mask.dim() != 4 or tuple(block_mask.shape[2:]) != (T, T) or block_mask.shape[0] not in (1, B) or \
            block_mask.shape[1] not in (1, Hq):
        raise ValueError(f"block_mask must be [B or 1, Hq or 1, {T}, {T}]")
    if block_mask.stride(3) != 1 or block_mask.stride(2) != T:
        raise ValueError("the last two dimensions of block_mask must be dense")
    sb = 0 if block_mask.shape[0] == 1 else block_mask.stride(0)
    sh = 0 if block_mask.shape[1] == 1 else block_mask.stride(1)
    return _ptr(block_mask), sb, sh


def fwd(q, k, v, causal=False, scale=None, out=None, lse=None, block_mask=None):
    """O, LSE = attention(q, k, v) on the current stream.

    q: [B, Hq, N, d]; k, v: [B, Hkv, N, d]; bf16 (fa_fwd) or fp32 (fa_fwd_f32)
    contiguous CUDA tensors. block_mask (bf16 only): uint8/bool
    [B or 1, Hq or 1, T, T], T = ceil(N/128), nonzero where query tile i may
    see key tile j (fa_fwd_blocksparse). k and v may hold another number of
    positions Nk than q (bf16, fa_fwd_kv: the queries are the last N of Nk
    positions for the causal rule). Returns (o like q, lse fp32 [B, Hq, N])."""
    import torch
    lib = load()
    B, Hq, Hkv, N, d = _shape(q, k)
    if scale is None:
        scale = d ** -0.5
    Nk = k.shape[2]
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q, k, v must be bf16 or fp32")
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _require(q.device, (q, "q", q.dtype, (B, Hq, N, d)), (k, "k", q.dtype, (B, Hkv, Nk, d)),
             (v, "v", q.dtype, (B, Hkv, Nk, d)), (o, "out", q.dtype, (B, Hq, N, d)),
             (lse, "lse", torch.float32, (B, Hq, N)))
    if Nk != N:
        if q.dtype != torch.bfloat16 or block_mask is not None:
            raise ValueError("keys of another length need bf16 inputs and no block mask")
        _check("fa_fwd_kv", lib.fa_fwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, Nk, d,
                                          int(bool(causal)), float(scale), _stream(q)))
        return o, lse
    if block_mask is not None:
        if q.dtype != torch.bfloat16:
            raise ValueError("block masks need bf16 inputs")
        mp, sb, sh = _mask_args(block_mask, B, Hq, N, q.device)
        _check("fa_fwd_blocksparse", lib.fa_fwd_blocksparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), mp, sb, sh,
                                                            B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                                                            _stream(q)))
        return o, lse
    fn = {torch.bfloat16: "fa_fwd", torch.float32: "fa_fwd_f32"}.get(q.dtype)
    if fn is None:
        raise ValueError("dtype must be bfloat16 or float32")
    _check(fn, getattr(lib, fn)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                B, Hq, Hkv, N, d, int(bool(causal)), float(scale), _stream(q)))
    return o, lse


def quantize_fp8(q, k, v):
    """Block-scaled e4m3 copies of bf16 q [B, Hq, N, d], k and v [B, Hkv, Nk, d] (fa_fp8_quantize_rows,
    fa_fp8_quantize_v): returns (q8, q_scale, k8, k_scale, vt8, v_scale) with
    q8, k8 uint8 [B, H, N, d], scales fp32 [B, H, ceil(N/64)], vt8 uint8
    [B, Hkv, d, NP] (V transposed, NP = N rounded up to 128) and v_scale
    fp32 [B, Hkv, d]."""
    import torch
    lib = load()
    B, Hq, Hkv, N, d = _shape(q, k)
    Nk = k.shape[2]
    bf16 = torch.bfloat16
    _require(q.device, (q, "q", bf16, (B, Hq, N, d)), (k, "k", bf16, (B, Hkv, Nk, d)), (v, "v", bf16, (B, Hkv, Nk, d)))
    nb, nbk, NP = int(lib.fa_fp8_row_scales(N)), int(lib.fa_fp8_row_scales(Nk)), int(lib.fa_fp8_vt_keys(Nk))
    dev = q.device
    q8 = torch.empty(q.shape, dtype=torch.uint8, device=dev)
    k8 = torch.empty(k.shape, dtype=torch.uint8, device=dev)
    vt8 = torch.empty((B, Hkv, d, NP), dtype=torch.uint8, device=dev)
    qs = torch.empty((B, Hq, nb), dtype=torch.float32, device=dev)
    ks = torch.empty((B, Hkv, nbk), dtype=torch.float32, device=dev)
    vs = torch.empty((B, Hkv, d), dtype=torch.float32, device=dev)
    st = _stream(q)
    _check("fa_fp8_quantize_rows", lib.fa_fp8_quantize_rows(_ptr(q), _ptr(q8), _ptr(qs), B * Hq, N, d, st))
    _check("fa_fp8_quantize_rows", lib.fa_fp8_quantize_rows(_ptr(k), _ptr(k8), _ptr(ks), B * Hkv, Nk, d, st))
    _check("fa_fp8_quantize_v", lib.fa_fp8_quantize_v(_ptr(v), _ptr(vt8), _ptr(vs), B * Hkv, Nk, d, st))
    return q8, qs, k8, ks, vt8, vs


def fwd_fp8(q8, q_scale, k8, k_scale, vt8, v_scale, causal=False, scale=None, out=None, lse=None):
    """O (bf16), LSE = attention of block-scaled e4m3 inputs (fa_fwd_fp8), as
    returned by quantize_fp8."""
    import torch
    lib = load()
    B, Hq, Hkv, N, d = _shape(q8, k8)
    Nk = k8.shape[2]
    dev = q8.device
    if scale is None:
        scale = d ** -0.5
    o = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device=dev) if out is None else out
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev) if lse is None else lse
    f32, u8 = torch.float32, torch.uint8
    _require(dev, (q8, "q8", u8, (B, Hq, N, d)), (q_scale, "q_scale", f32, (B, Hq, int(lib.fa_fp8_row_scales(N)))),
             (k8, "k8", u8, (B, Hkv, Nk, d)), (k_scale, "k_scale", f32, (B, Hkv, int(lib.fa_fp8_row_scales(Nk)))),
             (vt8, "vt8", u8, (B, Hkv, d, int(lib.fa_fp8_vt_keys(Nk)))), (v_scale, "v_scale", f32, (B, Hkv, d)),
             (o, "out", torch.bfloat16, (B, Hq, N, d)), (lse, "lse", f32, (B, Hq, N)))
    if Nk != N:
        # queries are the last N of Nk positions (fa_fwd_fp8_kv)
        _check("fa_fwd_fp8_kv", lib.fa_fwd_fp8_kv(_ptr(q8), _ptr(q_scale), _ptr(k8), _ptr(k_scale), _ptr(vt8),
                                                  _ptr(v_scale), _ptr(o), _ptr(lse), B, Hq, Hkv, N, Nk, d,
                                                  int(bool(causal)), float(scale), _stream(q8)))
        return o, lse
    _check("fa_fwd_fp8", lib.fa_fwd_fp8(_ptr(q8), _ptr(q_scale), _ptr(k8), _ptr(k_scale), _ptr(vt8), _ptr(v_scale),
                                        _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
                                        _stream(q8)))
    return o, lse


def bwd_workspace_bytes(B, Hq, Hkv, N, d):
    return int(load().fa_bwd_workspace_bytes(B, Hq, Hkv, N, d))


def bwd(q, k, v, o, lse, do, causal=False, scale=None, workspace=None, dq=None, dk=None, dv=None,
        deterministic=False, block_mask=None):
    """dQ, dK, dV of <O, dO> on the current stream (bf16 tensors, fp32 lse).

    deterministic=True runs fa_bwd_deterministic (bit-reproducible, slower);
    block_mask (as in fwd) runs fa_bwd_blocksparse."""
    import torch
    lib = load()
    B, Hq, Hkv, N, d = _shape(q, k)
    if scale is None:
        scale = d ** -0.5
    Nk = k.shape[2]
    dev = q.device
    bf16 = torch.bfloat16
    if block_mask is not None and deterministic:
        raise ValueError("the deterministic backward has no block-sparse form")
    if Nk != N and (deterministic or block_mask is not None):
        raise ValueError("keys of another length: only the default backward")
    nbytes = (int(lib.fa_bwd_blocksparse_workspace_bytes(B, Hq, Hkv, N, d)) if block_mask is not None
              else bwd_workspace_bytes(B, Hq, Hkv, N, d))
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    # the workspace's byte count is passed on; the library refuses one that is too small
    _require(dev, (q, "q", bf16, (B, Hq, N, d)), (k, "k", bf16, (B, Hkv, Nk, d)), (v, "v", bf16, (B, Hkv, Nk, d)),
             (o, "o", bf16, (B, Hq, N, d)), (lse, "lse", torch.float32, (B, Hq, N)), (do, "do", bf16, (B, Hq, N, d)),
             (workspace, "workspace", torch.uint8, (workspace.numel(),)), (dq, "dq", bf16, (B, Hq, N, d)),
             (dk, "dk", bf16, (B, Hkv, Nk, d)), (dv, "dv", bf16, (B, Hkv, Nk, d)))
    if Nk != N:
        _check("fa_bwd_kv", lib.fa_bwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                                          _ptr(dv), _ptr(workspace), workspace.numel(), B, Hq, Hkv, N, Nk, d,
                                          int(bool(causal)), float(scale), _stream(q)))
        return dq, dk, dv
    if block_mask is not None:
        mp, sb, sh = _mask_args(block_mask, B, Hq, N, q.device)
        _check("fa_bwd_blocksparse", lib.fa_bwd_blocksparse(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
            _ptr(workspace), workspace.numel(), mp, sb, sh, B, Hq, Hkv, N, d, int(bool(causal)), float(scale),
            _stream(q)))
        return dq, dk, dv
    name = "fa_bwd_deterministic" if deterministic else "fa_bwd"
    _check(name, getattr(lib, name)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                    _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(),
                                    B, Hq, Hkv, N, d, int(bool(causal)), float(scale), _stream(q)))
    return dq, dk, dv


def ex2_throughput(stream=None):
    """ex2 results per SM clock cycle on the current device (fa_ex2_throughput):
    the rate behind the forward's exponential ceiling."""
    import torch
    s = ctypes.c_void_p(stream if stream is not None else torch.cuda.current_stream().cuda_stream)
    out = ctypes.c_double(0.0)
    _check("fa_ex2_throughput", load().fa_ex2_throughput(ctypes.byref(out), s))
    return out.value


def sm_clock_mhz(stream=None):
    """Mean SM clock (MHz) of the forward and dK/dV kernels since the last
    call, measured by the kernels (fa_sm_clock_mhz); 0.0 if none ran."""
    import torch
    s = ctypes.c_void_p(stream if stream is not None else torch.cuda.current_stream().cuda_stream)
    out = ctypes.c_double(0.0)
    _check("fa_sm_clock_mhz", load().fa_sm_clock_mhz(ctypes.byref(out), s))
    return out.value


def check_device_status(stream=None):
    """Synchronise the stream and raise if a kernel's bounded wait ran out."""
    import torch
    s = ctypes.c_void_p(stream if stream is not None else torch.cuda.current_stream().cuda_stream)
    _check("fa_device_status", load().fa_device_status(s))
