"""ctypes binding of libgemm_f32.so (argument marshalling only).

Every step of the multiply runs in the library's CUDA kernels.  This module
turns torch CUDA tensors into the pointers, sizes, leading dimensions and
stream handle that ``include/gemm_f32.h`` declares, checks the returned
status, and raises ``GemmError`` on failure.  PyTorch serves only as the
owner of device memory and streams.
"""

from __future__ import annotations

import ctypes
import os
import threading

ALGO_AUTO, ALGO_SIMT, ALGO_TMA, ALGO_TF32X3 = 0, 1, 2, 3
ALGO_NAMES = {ALGO_AUTO: "auto", ALGO_SIMT: "simt", ALGO_TMA: "tma",
              ALGO_TF32X3: "tf32x3"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def library_path() -> str:
    return os.environ.get("GEMM_F32_LIBRARY",
                          os.path.join(_HERE, "libgemm_f32.so"))


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"libgemm_f32.so not found at {path}: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(path)
        i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        args = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp]
        L.gemm_f32.restype = ci
        L.gemm_f32.argtypes = args
        L.gemm_f32_ex.restype = ci
        L.gemm_f32_ex.argtypes = args + [ci]
        L.gemm_f32_ws.restype = ci
        L.gemm_f32_ws.argtypes = args[:-1] + [vp, i64, vp]
        L.gemm_f32_bias_act.restype = ci
        L.gemm_f32_bias_act.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp,
                                        ci, vp, i64, vp, i64, vp]
        L.gemm_f32_batched.restype = ci
        L.gemm_f32_batched.argtypes = [ci, ci, i64, i64, i64, vp, i64, i64,
                                       vp, i64, i64, vp, i64, i64, i64, vp]
        L.gemm_f32_plan.restype = ci
        L.gemm_f32_plan.argtypes = args[:-1] + [ctypes.POINTER(i64)]
        L.gemm_f32_batched_ws.restype = ci
        L.gemm_f32_batched_ws.argtypes = [ci, ci, i64, i64, i64, vp, i64,
                                          i64, vp, i64, i64, vp, i64, i64,
                                          i64, vp, i64, vp]
        L.gemm_f32_batched_workspace_size.restype = i64
        L.gemm_f32_batched_workspace_size.argtypes = [ci, ci, i64, i64, i64,
                                                      i64]
        L.gemm_f32_host.restype = ci
        L.gemm_f32_host.argtypes = args[:-1] + [vp, vp, vp, vp, i64, vp]
        L.gemm_f32_noalloc.restype = ci
        L.gemm_f32_noalloc.argtypes = args
        L.gemm_f32_noalloc_scratch_bytes.restype = i64
        L.gemm_f32_noalloc_scratch_bytes.argtypes = []
        L.gemm_f32_workspace_size.restype = i64
        L.gemm_f32_workspace_size.argtypes = [i64, i64, i64]
        L.gemm_f32_select_algo.restype = ci
        L.gemm_f32_select_algo.argtypes = args[:-1]
        L.gemm_f32_status_string.restype = ctypes.c_char_p
        L.gemm_f32_status_string.argtypes = [ci]
        L.gemm_f32_last_cuda_error.restype = ci
        L.gemm_f32_last_cuda_error.argtypes = []
        L.gemm_f32_device_status.restype = ci
        L.gemm_f32_device_status.argtypes = [vp]
        L.gemm_f32_set_wait_timeout_ns.restype = i64
        L.gemm_f32_set_wait_timeout_ns.argtypes = [i64]
        L.gemm_f32_set_debug_flags.restype = ctypes.c_uint
        L.gemm_f32_set_debug_flags.argtypes = [ctypes.c_uint]
        L.gemm_f32_version.restype = ci
        L.gemm_f32_version.argtypes = []
        L.gemm_f32_bounds_checked.restype = ci
        L.gemm_f32_bounds_checked.argtypes = []
        L.gemm_f32_bounds_probe.restype = ci
        L.gemm_f32_bounds_probe.argtypes = [vp]
        L.gemm_f32_mixed16.restype = ci
        L.gemm_f32_mixed16.argtypes = [ci, i64, i64, i64, vp, i64, vp, i64,
                                       vp, i64, vp]
        L.gemm_f32_mixed.restype = ci
        L.gemm_f32_mixed.argtypes = [ci, i64, i64, i64, vp, i64, vp, i64, vp,
                                     i64, vp, i64, vp]
        L.gemm_f32_round16.restype = ci
        L.gemm_f32_round16.argtypes = [ci, i64, i64, vp, i64, vp, i64, vp]
        L.gemm_f32_ffma_peak_launch.restype = ci
        L.gemm_f32_ffma_peak_launch.argtypes = [i64, vp, vp]
        L.gemm_f32_ffma_peak_flops.restype = i64
        L.gemm_f32_ffma_peak_flops.argtypes = [i64]
        L.gemm_f32_mixed_workspace_size.restype = i64
        L.gemm_f32_mixed_workspace_size.argtypes = [i64, i64, i64]
        L.gemm_f32_mixed_plan.restype = ci
        L.gemm_f32_mixed_plan.argtypes = [i64, i64, i64, ctypes.POINTER(i64)]
        L.gemm_f32_plan_sms.restype = ci
        L.gemm_f32_plan_sms.argtypes = args[:-1] + [ci, ci,
                                                    ctypes.POINTER(i64)]
        L.gemm_f32_mixed_plan_sms.restype = ci
        L.gemm_f32_mixed_plan_sms.argtypes = [i64, i64, i64, ci,
                                              ctypes.POINTER(i64)]
        L.gemm_f32_host_chunks.restype = ci
        L.gemm_f32_host_chunks.argtypes = [i64, i64, ci, ctypes.POINTER(i64)]
        _lib = L
        return L


def status_string(status: int) -> str:
    return lib().gemm_f32_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != 0:
        L = lib()
        msg = f"{what}: {status_string(status)}"
        if status == 3:
            msg += f" (cudaError {L.gemm_f32_last_cuda_error()})"
        raise GemmError(status, msg)


def gemm_f32_ptr(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, stream=0,
                 algo=ALGO_AUTO):
    """Raw-pointer call; device addresses and the stream handle as ints."""
    st = lib().gemm_f32_ex(int(M), int(N), int(K), a_ptr or None, int(lda),
                           b_ptr or None, int(ldb), c_ptr or None, int(ldc),
                           stream or None, int(algo))
    _check(st, "gemm_f32")


def gemm_f32_ws_ptr(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, ws_ptr,
                    ws_bytes, stream=0):
    """Raw-pointer gemm_f32_ws call (automatic kernel, optional scratch)."""
    st = lib().gemm_f32_ws(int(M), int(N), int(K), a_ptr or None, int(lda),
                           b_ptr or None, int(ldb), c_ptr or None, int(ldc),
                           ws_ptr or None, int(ws_bytes), stream or None)
    _check(st, "gemm_f32_ws")


def gemm_f32_noalloc_ptr(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc,
                         stream=0):
    """Raw-pointer gemm_f32_noalloc call: split-K scratch is the library's
    own static buffer, so nothing is allocated (for callers that may not
    allocate device memory)."""
    st = lib().gemm_f32_noalloc(int(M), int(N), int(K), a_ptr or None,
                                int(lda), b_ptr or None, int(ldb),
                                c_ptr or None, int(ldc), stream or None)
    _check(st, "gemm_f32_noalloc")


OP_N, OP_T = 0, 1
ACT_NONE, ACT_GELU = 0, 1


def gemm_f32_bias_act_ptr(M, N, K, a_ptr, lda, b_ptr, ldb, bias_ptr, act,
                          c_ptr, ldc, ws_ptr=0, ws_bytes=0, stream=0):
    """Raw-pointer gemm_f32_bias_act call."""
    st = lib().gemm_f32_bias_act(int(M), int(N), int(K), a_ptr or None,
                                 int(lda), b_ptr or None, int(ldb),
                                 bias_ptr or None, int(act), c_ptr or None,
                                 int(ldc), ws_ptr or None, int(ws_bytes),
                                 stream or None)
    _check(st, "gemm_f32_bias_act")


def gemm_f32_bias_act(a, b, bias=None, act=ACT_NONE, c=None, workspace=None,
                      stream=None):
    """C = act(A·B + bias) on CUDA tensors (bias: length-N or None)."""
    import torch
    M, K, ap, lda = _matrix_args(a, "a")
    K2, N, bp, ldb = _matrix_args(b, "b")
    if K != K2:
        raise ValueError("inner sizes differ")
    if c is None:
        c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    Mc, Nc, cp, ldc = _matrix_args(c, "c")
    if (Mc, Nc) != (M, N):
        raise ValueError("c has the wrong shape")
    bias_ptr = 0
    if bias is not None:
        if not bias.is_cuda or bias.dtype != torch.float32 or \
                bias.numel() != N or (N > 1 and bias.stride(-1) != 1):
            raise ValueError("bias must be a contiguous float32 CUDA vector "
                             "of N elements")
        bias_ptr = bias.data_ptr()
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        ws_bytes = workspace.numel() * workspace.element_size()
        ws_ptr = workspace.data_ptr() if ws_bytes else 0
    if stream is None:
        stream = torch.cuda.current_stream(a.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    with torch.cuda.device(a.device):
        st = lib().gemm_f32_bias_act(M, N, K, ap or None, lda, bp or None,
                                     ldb, bias_ptr or None, int(act),
                                     cp or None, ldc, ws_ptr or None, ws_bytes,
                                     handle or None)
    _check(st, "gemm_f32_bias_act")
    return c


def gemm_f32_batched_ptr(opA, opB, M, N, K, a_ptr, lda, sA, b_ptr, ldb, sB,
                         c_ptr, ldc, sC, batch, stream=0):
    """Raw-pointer gemm_f32_batched call."""
    st = lib().gemm_f32_batched(int(opA), int(opB), int(M), int(N), int(K),
                                a_ptr or None, int(lda), int(sA),
                                b_ptr or None, int(ldb), int(sB),
                                c_ptr or None, int(ldc), int(sC), int(batch),
                                stream or None)
    _check(st, "gemm_f32_batched")


def gemm_f32_batched_ws_ptr(opA, opB, M, N, K, a_ptr, lda, sA, b_ptr, ldb,
                            sB, c_ptr, ldc, sC, batch, ws_ptr, ws_bytes,
                            stream=0):
    """Raw-pointer gemm_f32_batched_ws call (optional scratch)."""
    st = lib().gemm_f32_batched_ws(int(opA), int(opB), int(M), int(N),
                                   int(K), a_ptr or None, int(lda), int(sA),
                                   b_ptr or None, int(ldb), int(sB),
                                   c_ptr or None, int(ldc), int(sC),
                                   int(batch), ws_ptr or None, int(ws_bytes),
                                   stream or None)
    _check(st, "gemm_f32_batched_ws")


def batched_workspace_size(opA, opB, M, N, K, batch=1) -> int:
    """Scratch bytes gemm_f32_batched_ws uses at most."""
    n = int(lib().gemm_f32_batched_workspace_size(int(opA), int(opB), int(M),
                                                  int(N), int(K), int(batch)))
    if n < 0:
        _check(-n, "gemm_f32_batched_workspace_size")
    return n


def _scratch(nbytes, device, stream):
    """A device byte buffer for one call on `stream` (a torch stream, a raw
    handle or None = current).  The caching allocator is told when the
    stream is not the current one, so that the buffer is not handed out
    again while that stream may still use it."""
    import torch
    buf = torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)
    if stream is None:
        return buf
    current = torch.cuda.current_stream(device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") \
        else int(stream)
    if handle == current.cuda_stream:
        return buf
    if isinstance(stream, torch.cuda.Stream):
        buf.record_stream(stream)
    elif handle == 0:
        buf.record_stream(torch.cuda.default_stream(device))
    else:
        buf.record_stream(torch.cuda.ExternalStream(handle, device=device))
    return buf


def gemm_f32_batched(a, b, c=None, trans_a=False, trans_b=False,
                     stream=None, workspace=None):
    """C[i] = op(A[i]) · op(B[i]) for 3-D CUDA tensors (batch, rows, cols).

    op(X) is X or, with trans_*, X transposed (read in place, no copy).  A
    2-D operand is used for every product (stride 0).  For op(A) = Aᵀ with
    op(B) = B the call goes through gemm_f32_batched_ws with `workspace`
    (a CUDA tensor; allocated here when None) holding a transposed copy of
    A; other forms use `workspace` only when given.
    """
    import torch

    def views(t, name):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or \
                not t.is_cuda:
            raise TypeError(f"{name} must be a float32 CUDA tensor")
        if t.dim() == 2:
            t = t.unsqueeze(0).expand(1, *t.shape)
            stride0 = 0
        elif t.dim() == 3:
            stride0 = t.stride(0) if t.shape[0] > 1 else 0
        else:
            raise ValueError(f"{name} must be 2-D or 3-D")
        rows, cols = t.shape[1], t.shape[2]
        if cols > 1 and t.stride(2) != 1:
            raise ValueError(f"{name} must be row-major")
        ld = t.stride(1) if rows > 1 else max(cols, 1)
        return t, rows, cols, max(ld, cols, 1), stride0

    a3, ar, ac, lda, sA = views(a, "a")
    b3, br, bc, ldb, sB = views(b, "b")
    M, K = (ac, ar) if trans_a else (ar, ac)
    K2, N = (bc, br) if trans_b else (br, bc)
    if K != K2:
        raise ValueError("inner sizes differ")
    batch = max(a3.shape[0] if a.dim() == 3 else 1,
                b3.shape[0] if b.dim() == 3 else 1)
    if c is None:
        c = torch.empty((batch, M, N), dtype=torch.float32, device=a.device)
    c3, cr, cc, ldc, sC = views(c, "c")
    if (cr, cc) != (M, N) or (c.dim() == 3 and c.shape[0] != batch):
        raise ValueError("c has the wrong shape")
    if batch > 1 and sC == 0:
        raise ValueError("c must hold one matrix per product")
    opa, opb = (OP_T if trans_a else OP_N), (OP_T if trans_b else OP_N)
    _batched_call(opa, opb, M, N, K, a3.data_ptr(), lda, sA, b3.data_ptr(),
                  ldb, sB, c3.data_ptr(), ldc, sC, batch, a.device, stream,
                  workspace)
    return c


def _batched_call(opa, opb, M, N, K, ap, lda, sA, bp, ldb, sB, cp, ldc, sC,
                  batch, device, stream, workspace):
    """gemm_f32_batched_ws with the given scratch, or with scratch allocated
    for the Aᵀ·B form, else gemm_f32_batched."""
    import torch
    with torch.cuda.device(device):
        handle = _handle(stream, device)
        if workspace is None and opa == OP_T and opb == OP_N:
            need = batched_workspace_size(opa, opb, M, N, K, batch)
            if need > 0:
                workspace = _scratch(need, device, stream)
        if workspace is None:
            gemm_f32_batched_ptr(opa, opb, M, N, K, ap, lda, sA, bp, ldb, sB,
                                 cp, ldc, sC, batch, handle)
            return
        if not workspace.is_cuda:
            raise ValueError("workspace must live on a CUDA device")
        nbytes = workspace.numel() * workspace.element_size()
        gemm_f32_batched_ws_ptr(opa, opb, M, N, K, ap, lda, sA, bp, ldb, sB,
                                cp, ldc, sC, batch,
                                workspace.data_ptr() if nbytes else 0, nbytes,
                                handle)


def gemm_f32_host(a, b, c, da, db, dc, workspace=None, stream=None):
    """C = A·B for CPU tensors a, b, c (pin them for overlapped copies),
    through caller-lent CUDA buffers da (M×K), db (K×N), dc (M×N),
    contiguous.  Copies, multiply and copy-back overlap in row chunks."""
    import torch
    for t, name in ((a, "a"), (b, "b"), (c, "c")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or \
                t.dim() != 2 or t.is_cuda:
            raise TypeError(f"{name} must be a 2-D float32 CPU tensor")
        if t.numel() and t.shape[1] > 1 and t.stride(1) != 1:
            raise ValueError(f"{name} must be row-major")
    M, K = a.shape
    K2, N = b.shape
    if K != K2 or tuple(c.shape) != (M, N):
        raise ValueError("shape mismatch")
    for t, shape, name in ((da, (M, K), "da"), (db, (K, N), "db"),
                           (dc, (M, N), "dc")):
        if not t.is_cuda or not t.is_contiguous() or \
                t.numel() < shape[0] * shape[1]:
            raise ValueError(f"{name} must be a contiguous CUDA buffer of "
                             f"at least {shape[0]}x{shape[1]} floats")
    if stream is None:
        stream = torch.cuda.current_stream(dc.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream

    def ld(t, cols):
        return max(t.stride(0) if t.shape[0] > 1 else cols, cols, 1)

    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        ws_bytes = workspace.numel() * workspace.element_size()
        ws_ptr = workspace.data_ptr() if ws_bytes else 0
    with torch.cuda.device(dc.device):
        st = lib().gemm_f32_host(
            M, N, K, a.data_ptr() or None, ld(a, K), b.data_ptr() or None,
            ld(b, N), c.data_ptr() or None, ld(c, N), da.data_ptr() or None,
            db.data_ptr() or None, dc.data_ptr() or None, ws_ptr or None,
            ws_bytes, handle or None)
    _check(st, "gemm_f32_host")
    return c


def noalloc_scratch_bytes() -> int:
    """Capacity of the static scratch buffer gemm_f32_noalloc uses."""
    return int(lib().gemm_f32_noalloc_scratch_bytes())


def workspace_size(M, N, K) -> int:
    """Scratch bytes gemm_f32_ws would use for aligned M×N×K operands."""
    n = int(lib().gemm_f32_workspace_size(int(M), int(N), int(K)))
    if n < 0:
        _check(-n, "gemm_f32_workspace_size")
    return n


def _matrix_args(t, name, dtypes=None):
    import torch
    dtypes = dtypes or (torch.float32,)
    if not isinstance(t, torch.Tensor) or t.dtype not in dtypes:
        names = " or ".join(str(d).replace("torch.", "") for d in dtypes)
        raise TypeError(f"{name} must be a {names} torch tensor")
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    rows, cols = t.shape
    if t.numel() == 0:
        return rows, cols, 0, max(cols, 1)
    if cols > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major (unit column stride)")
    # a single row has no meaningful row stride unless it spans the width
    ld = t.stride(0) if (rows > 1 or t.stride(0) >= cols) else cols
    return rows, cols, t.data_ptr(), max(ld, cols, 1)


def gemm_f32_ex(a, b, c=None, algo=ALGO_AUTO, stream=None):
    """C = A·B on torch CUDA tensors; returns C (allocated if not given)."""
    import torch
    M, K, ap, lda = _matrix_args(a, "a")
    K2, N, bp, ldb = _matrix_args(b, "b")
    if K != K2:
        raise ValueError(f"inner sizes differ: {tuple(a.shape)} x "
                         f"{tuple(b.shape)}")
    if c is None:
        c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    Mc, Nc, cp, ldc = _matrix_args(c, "c")
    if (Mc, Nc) != (M, N):
        raise ValueError(f"c has shape {tuple(c.shape)}, want {(M, N)}")
    if stream is None:
        stream = torch.cuda.current_stream(a.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    with torch.cuda.device(a.device):
        gemm_f32_ptr(M, N, K, ap, lda, bp, ldb, cp, ldc, handle, algo)
    return c


def gemm_f32(a, b, c=None, stream=None, workspace=None):
    """C = A·B with the automatically selected kernel.

    ``workspace``: optional CUDA tensor used as split-K scratch through
    gemm_f32_ws (see ``workspace_size``); None runs gemm_f32 without it.
    """
    if workspace is None:
        return gemm_f32_ex(a, b, c, ALGO_AUTO, stream)
    import torch
    M, K, ap, lda = _matrix_args(a, "a")
    K2, N, bp, ldb = _matrix_args(b, "b")
    if K != K2:
        raise ValueError(f"inner sizes differ: {tuple(a.shape)} x "
                         f"{tuple(b.shape)}")
    if c is None:
        c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    Mc, Nc, cp, ldc = _matrix_args(c, "c")
    if (Mc, Nc) != (M, N):
        raise ValueError(f"c has shape {tuple(c.shape)}, want {(M, N)}")
    if not workspace.is_cuda:
        raise ValueError("workspace must live on a CUDA device")
    if stream is None:
        stream = torch.cuda.current_stream(a.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    nbytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(a.device):
        gemm_f32_ws_ptr(M, N, K, ap, lda, bp, ldb, cp, ldc,
                        workspace.data_ptr() if nbytes else 0, nbytes, handle)
    return c


def plan(M, N, K, a_ptr=16, lda=None, b_ptr=16, ldb=None, c_ptr=16,
         ldc=None, sm_count=None, cc_major=10) -> dict:
    """The automatic plan for these sizes (default: 16-byte aligned
    pointers, leading dimensions = the row widths rounded up to multiples
    of 4, the layouts the tensor kernels take): kernel family, tensor
    variant ("tiled" / "streaming"), split-K ways, whole tiles, rows of C
    per tensor tile (0 for the FFMA kernels).  On the current device, or,
    with `sm_count` given, on a device of that many SMs and compute
    capability major `cc_major` without any CUDA call."""
    def pad4(x):
        return max((int(x) + 3) // 4 * 4, 4)
    out = (ctypes.c_int64 * 5)()
    args = (int(M), int(N), int(K), a_ptr or None,
            int(lda if lda is not None else pad4(K)), b_ptr or None,
            int(ldb if ldb is not None else pad4(N)), c_ptr or None,
            int(ldc if ldc is not None else pad4(N)))
    if sm_count is None:
        _check(lib().gemm_f32_plan(*args, out), "gemm_f32_plan")
    else:
        _check(lib().gemm_f32_plan_sms(*args, int(sm_count), int(cc_major),
                                       out), "gemm_f32_plan_sms")
    return {"algo": out[0], "variant": "streaming" if out[1] else "tiled",
            "splits": out[2], "whole_tiles": out[3], "tile_rows": out[4]}


def select_algo(M, N, K, a_ptr=0, lda=None, b_ptr=0, ldb=None, c_ptr=0,
                ldc=None) -> int:
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    return int(lib().gemm_f32_select_algo(M, N, K, a_ptr or None, lda,
                                          b_ptr or None, ldb, c_ptr or None,
                                          ldc))


def device_status(stream=None) -> int:
    """Waits for the stream, returns and clears the kernels' status word."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    return int(lib().gemm_f32_device_status(handle or None))


def set_wait_timeout_ns(ns: int) -> int:
    return int(lib().gemm_f32_set_wait_timeout_ns(int(ns)))


def set_debug_flags(flags: int) -> int:
    return int(lib().gemm_f32_set_debug_flags(int(flags)))


DEBUG_STALL_PRODUCER = 1


def bounds_checked() -> bool:
    """True when the loaded library is the checked build."""
    return bool(lib().gemm_f32_bounds_checked())


def bounds_probe(stream=None):
    """Checked build: makes the next device_status() report
    GEMM_F32_ERR_BOUNDS (no memory is touched); no-op otherwise."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    _check(lib().gemm_f32_bounds_probe(handle or None), "gemm_f32_bounds_probe")


def version() -> int:
    return int(lib().gemm_f32_version())


# ------------------------------------------------ mixed precision (16-bit)
MIXED_BF16, MIXED_F16 = 0, 1


def _mixed_type(dtype_or_type):
    import torch
    if dtype_or_type in (MIXED_BF16, torch.bfloat16):
        return MIXED_BF16
    if dtype_or_type in (MIXED_F16, torch.float16):
        return MIXED_F16
    raise ValueError("16-bit type must be bfloat16 or float16")


def _mixed_dtype(t):
    import torch
    return torch.bfloat16 if t == MIXED_BF16 else torch.float16


def _handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def gemm_f32_mixed16_ptr(type_, M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc,
                         stream=0):
    """Raw-pointer gemm_f32_mixed16 call (16-bit operands, fp32 C)."""
    st = lib().gemm_f32_mixed16(int(type_), int(M), int(N), int(K),
                                a_ptr or None, int(lda), b_ptr or None,
                                int(ldb), c_ptr or None, int(ldc),
                                stream or None)
    _check(st, "gemm_f32_mixed16")


def gemm_f32_mixed16(a, b, c=None, stream=None):
    """C (fp32) = A·B for bfloat16 or float16 CUDA tensors of one dtype,
    fp32 accumulation on the tensor cores."""
    import torch
    if a.dtype != b.dtype:
        raise TypeError("a and b must have the same 16-bit dtype")
    dt = (torch.bfloat16, torch.float16)
    M, K, ap, lda = _matrix_args(a, "a", dt)
    K2, N, bp, ldb = _matrix_args(b, "b", dt)
    if K != K2:
        raise ValueError("inner sizes differ")
    if c is None:
        c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    Mc, Nc, cp, ldc = _matrix_args(c, "c")
    if (Mc, Nc) != (M, N):
        raise ValueError("c has the wrong shape")
    with torch.cuda.device(a.device):
        gemm_f32_mixed16_ptr(_mixed_type(a.dtype), M, N, K, ap, lda, bp, ldb,
                             cp, ldc, _handle(stream, a.device))
    return c


def round16_ptr(type_, rows, cols, src_ptr, lds, dst_ptr, ldd, stream=0):
    """Raw-pointer gemm_f32_round16 call."""
    st = lib().gemm_f32_round16(int(type_), int(rows), int(cols),
                                src_ptr or None, int(lds), dst_ptr or None,
                                int(ldd), stream or None)
    _check(st, "gemm_f32_round16")


def round16(x, half=MIXED_BF16, out=None, stream=None):
    """x (2-D float32 CUDA tensor) rounded to bfloat16 or float16 (nearest,
    ties to even) by the library's kernel; returns the 16-bit tensor."""
    import torch
    t = _mixed_type(half)
    rows, cols, xp, lds = _matrix_args(x, "x")
    if out is None:
        out = torch.empty((rows, cols), dtype=_mixed_dtype(t), device=x.device)
    r2, c2, op, ldd = _matrix_args(out, "out", (_mixed_dtype(t),))
    if (r2, c2) != (rows, cols):
        raise ValueError("out has the wrong shape")
    with torch.cuda.device(x.device):
        round16_ptr(t, rows, cols, xp, lds, op, ldd, _handle(stream, x.device))
    return out


def mixed_workspace_size(M, N, K) -> int:
    """Workspace bytes gemm_f32_mixed needs."""
    n = int(lib().gemm_f32_mixed_workspace_size(int(M), int(N), int(K)))
    if n < 0:
        _check(-n, "gemm_f32_mixed_workspace_size")
    return n


def mixed_plan(M, N, K=0, sm_count=None) -> dict:
    """How the 16-bit product cuts an M×N×K product on the current device
    (or, with `sm_count` given, on a device of that many SMs, without any
    CUDA call): tile width, tiles run whole, strips per remaining tile,
    CTAs, tile rows."""
    out = (ctypes.c_int64 * 5)()
    if sm_count is None:
        _check(lib().gemm_f32_mixed_plan(int(M), int(N), int(K), out),
               "gemm_f32_mixed_plan")
    else:
        _check(lib().gemm_f32_mixed_plan_sms(int(M), int(N), int(K),
                                             int(sm_count), out),
               "gemm_f32_mixed_plan_sms")
    return {"width": out[0], "whole": out[1], "parts": out[2], "grid": out[3],
            "rows": out[4]}


def host_chunks(M, N, sm_count) -> list:
    """The first row of each row chunk gemm_f32_host cuts an M×N product
    into on a device of `sm_count` SMs, then M (no CUDA call)."""
    bounds = (ctypes.c_int64 * 17)()
    n = lib().gemm_f32_host_chunks(int(M), int(N), int(sm_count), bounds)
    if n < 0:
        _check(-n, "gemm_f32_host_chunks")
    return [int(bounds[i]) for i in range(n + 1)]


def gemm_f32_mixed_ptr(type_, M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc,
                       ws_ptr, ws_bytes, stream=0):
    """Raw-pointer gemm_f32_mixed call (fp32 operands rounded first)."""
    st = lib().gemm_f32_mixed(int(type_), int(M), int(N), int(K),
                              a_ptr or None, int(lda), b_ptr or None,
                              int(ldb), c_ptr or None, int(ldc),
                              ws_ptr or None, int(ws_bytes), stream or None)
    _check(st, "gemm_f32_mixed")


def gemm_f32_mixed(a, b, half=MIXED_BF16, c=None, workspace=None,
                   stream=None):
    """Mixed-precision C = A·B of float32 CUDA tensors: operands rounded to
    bfloat16 (default) or float16, fp32 products and sums, fp32 C.  The
    rounding scratch is `workspace` (a CUDA tensor of at least
    mixed_workspace_size bytes), allocated here when not given."""
    import torch
    t = _mixed_type(half)
    M, K, ap, lda = _matrix_args(a, "a")
    K2, N, bp, ldb = _matrix_args(b, "b")
    if K != K2:
        raise ValueError("inner sizes differ")
    if c is None:
        c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    Mc, Nc, cp, ldc = _matrix_args(c, "c")
    if (Mc, Nc) != (M, N):
        raise ValueError("c has the wrong shape")
    need = mixed_workspace_size(M, N, K)
    if workspace is None:
        workspace = _scratch(need, a.device, stream)
    ws_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(a.device):
        gemm_f32_mixed_ptr(t, M, N, K, ap, lda, bp, ldb, cp, ldc,
                           workspace.data_ptr() if ws_bytes else 0, ws_bytes,
                           _handle(stream, a.device))
    return c


# ------------------------------------------------ FP32 FMA throughput probe
def ffma_peak_launch(iters, sink, stream=0):
    """Launches the FMA-chain probe (``sink``: a CUDA float32 tensor of at
    least 256 elements); time it on ``stream``."""
    st = lib().gemm_f32_ffma_peak_launch(int(iters), sink.data_ptr(),
                                         stream or None)
    _check(st, "gemm_f32_ffma_peak_launch")


def ffma_peak_flops(iters) -> int:
    n = int(lib().gemm_f32_ffma_peak_flops(int(iters)))
    if n < 0:
        _check(-n, "gemm_f32_ffma_peak_flops")
    return n


# ------------------------------------------------ layout-aware front end
def _operand_form(t, name):
    """(op, rows, cols, ld, batch, batch_stride) of a 2-D or 3-D float32
    CUDA tensor whose matrices are row-major (op N) or transposed views of
    row-major storage (op T, rows/cols of the logical matrix)."""
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or \
            not t.is_cuda:
        raise TypeError(f"{name} must be a float32 CUDA tensor")
    if t.dim() == 2:
        batch, sb = 1, 0
        r, c = t.shape
        s0, s1 = t.stride()
    elif t.dim() == 3:
        batch, r, c = t.shape
        sb = t.stride(0) if batch > 1 else 0
        s0, s1 = t.stride(1), t.stride(2)
    else:
        raise ValueError(f"{name} must be 2-D or 3-D")
    if s1 == 1 or c <= 1:
        return OP_N, r, c, max(s0 if r > 1 else c, c, 1), batch, sb
    if s0 == 1 or r <= 1:
        # element (i, j) at i + j·s1: the transpose of a c×r row-major
        # matrix with leading dimension s1
        return OP_T, r, c, max(s1 if c > 1 else r, r, 1), batch, sb
    raise ValueError(f"{name}: neither rows nor columns are contiguous; "
                     "pass a row-major tensor or a transposed view of one")


def matmul(a, b, out=None, stream=None):
    """The product a·b for float32 CUDA tensors, 2-D or batched 3-D (a 2-D
    operand is shared by every product), where each operand may be
    row-major or a transposed view of row-major storage (e.g. ``w.t()``):
    the library reads it in place through gemm_f32_batched (for a
    transposed ``a`` with a row-major ``b``, gemm_f32_batched_ws with a
    transposed copy of ``a`` in scratch allocated here).  Returns C
    (row-major, allocated if ``out`` is None)."""
    import torch
    opa, M, K, lda, ba, sa = _operand_form(a, "a")
    opb, K2, N, ldb, bb, sb = _operand_form(b, "b")
    if K != K2:
        raise ValueError(f"inner sizes differ: {tuple(a.shape)} x "
                         f"{tuple(b.shape)}")
    batch = max(ba, bb)
    if ba not in (1, batch) or bb not in (1, batch):
        raise ValueError("batch sizes differ")
    shape = (batch, M, N) if (a.dim() == 3 or b.dim() == 3) else (M, N)
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=a.device)
    elif tuple(out.shape) != shape or out.dtype != torch.float32:
        raise ValueError(f"out must be a float32 tensor of shape {shape}")
    opc, Mc, Nc, ldc, bc, sc = _operand_form(out, "out")
    if opc != OP_N:
        raise ValueError("out must be row-major")
    if batch > 1 and sc == 0:
        raise ValueError("out must hold one matrix per product")
    _batched_call(opa, opb, M, N, K, a.data_ptr(), lda, sa, b.data_ptr(),
                  ldb, sb, out.data_ptr(), ldc, sc, batch, a.device, stream,
                  None)
    return out
