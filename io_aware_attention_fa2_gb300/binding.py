"""ctypes binding over the C ABI in ``include/fa.h`` (argument marshalling only).

Every step of the attention forward runs in the CUDA library. This module turns torch tensors
into device pointers and sizes, calls the library, and turns nonzero status codes into
``FaError``. PyTorch only provides device memory and streams here.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libfa_gb300.so"

FA_BF16, FA_FP16 = 0, 1
FA_OK = 0
FA_ERR_TIMEOUT = -8

_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    """A nonzero status from the CUDA library."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (where, error_string(code), code))


def library_path() -> str:
    """The in-tree build, or the library named by FA_GB300_LIBRARY (another build of the same
    sources, e.g. with different compile flags)."""
    return os.environ.get("FA_GB300_LIBRARY") or os.path.join(_HERE, "_build", LIB_NAME)


def load_library() -> ctypes.CDLL:
    """Load the built CUDA library; raise if it has not been built. There is no fallback."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise FileNotFoundError(
                    "CUDA library %s is missing: build it with "
                    "io_aware_attention_fa2_gb300.build.build()" % path)
            lib = ctypes.CDLL(path)
            vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp]
            lib.fa_fwd.restype = i32
            lib.fa_fwd_masked.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                          vp, f32, i32, vp]
            lib.fa_fwd_masked.restype = i32
            lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                           i32, vp, f32, i32, i32, vp, ctypes.c_size_t, vp]
            lib.fa_fwd_splitkv.restype = i32
            lib.fa_fwd_splitkv_workspace_size.argtypes = [i32, i32, i32, i32, i32]
            lib.fa_fwd_splitkv_workspace_size.restype = ctypes.c_size_t
            lib.fa_fwd_splitkv_num_splits.argtypes = [i32, i32, i32, i32, i32]
            lib.fa_fwd_splitkv_num_splits.restype = i32
            lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                   f32, i32, vp, ctypes.c_size_t, vp]
            lib.fa_bwd.restype = i32
            lib.fa_bwd_masked.argtypes = [vp] * 9 + [i32] * 7 + [vp, f32, i32, vp,
                                                                 ctypes.c_size_t, vp]
            lib.fa_bwd_masked.restype = i32
            lib.fa_fwd_host.argtypes = [vp] * 10 + [i32, i32, i32, i32, i32, f32, i32, vp]
            lib.fa_fwd_host.restype = i32
            lib.fa_bwd_host.argtypes = [vp] * 19 + [ctypes.c_size_t] + [i32] * 5 + [f32, i32,
                                                                              vp]
            lib.fa_bwd_host.restype = i32
            lib.fa_fwd_host_masked.argtypes = [vp] * 10 + [i32] * 7 + [vp, f32, i32, vp]
            lib.fa_fwd_host_masked.restype = i32
            lib.fa_bwd_host_masked.argtypes = ([vp] * 19 + [ctypes.c_size_t] + [i32] * 7 +
                                               [vp, f32, i32, vp])
            lib.fa_bwd_host_masked.restype = i32
            lib.fa_bwd_workspace_size.argtypes = [i32, i32, i32, i32]
            lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
            lib.fa_error_string.argtypes = [i32]
            lib.fa_error_string.restype = ctypes.c_char_p
            lib.fa_get_device_error.argtypes = [vp]
            lib.fa_get_device_error.restype = i32
            lib.fa_selftest_wait_timeout.argtypes = [i32, vp]
            lib.fa_selftest_wait_timeout.restype = i32
            lib.fa_abi_version.argtypes = []
            lib.fa_abi_version.restype = i32
            _lib = lib
    return _lib


def available() -> bool:
    """True when the library is built and a CUDA device is visible."""
    try:
        import torch
        load_library()
        return torch.cuda.is_available()
    except (OSError, ImportError):
        return False


def error_string(code: int) -> str:
    try:
        return load_library().fa_error_string(int(code)).decode()
    except OSError:
        return "status %d" % code


def _stream_handle(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float16:
        return FA_FP16
    raise TypeError("q, k, v must be bfloat16 or float16, got %s" % t.dtype)


def fa_fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None, window=(-1, -1),
           seqlens_k=None) -> None:
    """Enqueue the attention forward on ``stream`` (default: torch's current stream).

    q, k, v, o: CUDA tensors [B, N, H, d] of one dtype (bf16/fp16), contiguous.
    lse: CUDA float32 tensor [B, H, N], contiguous.
    window: (left, right) sliding-window bounds (negative = none); seqlens_k: optional CUDA
    int32 tensor [B] of per-batch key lengths (padding mask). Either one selects
    ``fa_fwd_masked``; otherwise ``fa_fwd`` is called.
    """
    import torch
    if q.dim() != 4:
        raise ValueError("q must be [B, N, H, d]")
    B, N, H, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o)):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError("%s must match q's shape and dtype" % name)
    if lse.shape != (B, H, N) or lse.dtype != torch.float32:
        raise ValueError("lse must be float32 [B, H, N]")
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("lse", lse)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
    lib = load_library()
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
            int(bool(causal)))
    left, right = (int(w) for w in window)
    if seqlens_k is None and left < 0 and right < 0:
        rc = lib.fa_fwd(*args, float(scale), _dtype_code(q), _stream_handle(stream))
        where = "fa_fwd"
    else:
        lens_ptr = None
        if seqlens_k is not None:
            if (not seqlens_k.is_cuda or seqlens_k.dtype != torch.int32
                    or seqlens_k.shape != (B,) or not seqlens_k.is_contiguous()):
                raise ValueError("seqlens_k must be a contiguous CUDA int32 tensor [B]")
            lens_ptr = seqlens_k.data_ptr()
        rc = lib.fa_fwd_masked(*args, left, right, lens_ptr, float(scale), _dtype_code(q),
                               _stream_handle(stream))
        where = "fa_fwd_masked"
    if rc != FA_OK:
        raise FaError(rc, where)


def splitkv_workspace_size(B: int, H: int, Nq: int, d: int, num_splits: int) -> int:
    """Bytes of workspace fa_fwd_splitkv needs (0 for one part)."""
    return int(load_library().fa_fwd_splitkv_workspace_size(B, H, Nq, d, num_splits))


def splitkv_num_splits(B: int, H: int, Nq: int, Nk: int, num_sms: int | None = None) -> int:
    """The library's part count for fa_fwd_splitkv on a GPU with ``num_sms`` SMs (default:
    the current device's)."""
    if num_sms is None:
        import torch
        props = torch.cuda.get_device_properties(torch.cuda.current_device())
        num_sms = props.multi_processor_count
    return int(load_library().fa_fwd_splitkv_num_splits(B, H, Nq, Nk, num_sms))


def fa_fwd_splitkv(q, k, v, o, lse, causal: bool, scale: float, num_splits: int,
                   workspace=None, stream=None, window=(-1, -1), seqlens_k=None) -> None:
    """Enqueue the split-K/V forward: q, o [B, Nq, H, d]; k, v [B, Nk, H, d] (Nk >= Nq; the
    queries are the last Nq positions); lse float32 [B, H, Nq]. ``workspace``: a CUDA tensor of
    at least ``splitkv_workspace_size`` bytes, or None to let PyTorch allocate one (it must
    stay alive until the stream has run the call, which the caching allocator guarantees for
    the current stream)."""
    import torch
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be 4-D")
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    if k.shape != (B, Nk, H, d) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k, v must be [B, Nk, H, d] in q's dtype")
    if o.shape != q.shape or o.dtype != q.dtype:
        raise ValueError("o must match q")
    if lse.shape != (B, H, Nq) or lse.dtype != torch.float32:
        raise ValueError("lse must be float32 [B, H, Nq]")
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("lse", lse)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
    need = splitkv_workspace_size(B, H, Nq, d, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    lens_ptr = None
    if seqlens_k is not None:
        if (not seqlens_k.is_cuda or seqlens_k.dtype != torch.int32
                or seqlens_k.shape != (B,) or not seqlens_k.is_contiguous()):
            raise ValueError("seqlens_k must be a contiguous CUDA int32 tensor [B]")
        lens_ptr = seqlens_k.data_ptr()
    left, right = (int(w) for w in window)
    rc = load_library().fa_fwd_splitkv(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, d,
        int(bool(causal)), left, right, lens_ptr, float(scale), _dtype_code(q), int(num_splits),
        ws_ptr, ws_bytes, _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv")


def bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    """Bytes of workspace fa_bwd needs."""
    return int(load_library().fa_bwd_workspace_size(B, H, N, d))


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, causal: bool, scale: float, workspace=None,
           stream=None, window=(-1, -1), seqlens_k=None) -> None:
    """Enqueue the backward: dq, dk, dv [B, N, H, d] from the forward's q, k, v, o, lse and
    the upstream gradient dout. ``workspace``: a CUDA tensor of at least bwd_workspace_size
    bytes, or None to let PyTorch allocate one. ``window`` and ``seqlens_k`` (int32 CUDA
    tensor [B]) select the masks of fa_fwd_masked; lse must come from the forward with the
    same masks."""
    import torch
    B, N, H, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("dout", dout), ("dq", dq), ("dk", dk),
                    ("dv", dv)):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor like q" % name)
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be float32 [B, H, N]")
    need = bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    lens_ptr = None
    if seqlens_k is not None:
        if (not seqlens_k.is_cuda or seqlens_k.dtype != torch.int32
                or tuple(seqlens_k.shape) != (B,) or not seqlens_k.is_contiguous()):
            raise ValueError("seqlens_k must be a contiguous int32 CUDA tensor [B]")
        lens_ptr = seqlens_k.data_ptr()
    left, right = (int(w) for w in window)
    rc = load_library().fa_bwd_masked(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, int(bool(causal)), left, right,
        lens_ptr, float(scale), _dtype_code(q), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_masked")


def device_error(stream=None) -> int:
    """Synchronise ``stream`` and return-and-clear the device error word (0 = none)."""
    return int(load_library().fa_get_device_error(_stream_handle(stream)))


def attention_forward(q, k, v, causal: bool = False, scale: float | None = None, out=None,
                      lse=None, stream=None, device=None, window=(-1, -1), seqlens_k=None,
                      num_splits=None):
    """O, LSE = attention(q, k, v). The call a user makes.

    Device tensors are used in place. Host tensors (ideally pinned) are copied to ``device``
    (default cuda:0) on ``stream``, the kernel runs there, and O and LSE are copied back into
    host tensors, so the result is ready when the call returns. ``scale`` defaults to
    1/sqrt(d) rounded to fp32. ``window`` and ``seqlens_k`` (int32 [B], host or device) select
    the padding and sliding-window masks (see ``fa_fwd``). k and v may be longer than q (the
    queries are then the last positions, as when decoding); that case, or an explicit
    ``num_splits``, runs the split-K/V forward (``num_splits`` None: the library's choice).
    """
    import math

    import torch
    B, N, H, d = q.shape
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))
    split = num_splits is not None or k.shape[1] != N

    def run(qd, kd, vd, od, ld, st, lens):
        if split:
            ns = num_splits if num_splits is not None else splitkv_num_splits(
                B, H, N, kd.shape[1])
            fa_fwd_splitkv(qd, kd, vd, od, ld, causal, scale, ns, None, st, window, lens)
        else:
            fa_fwd(qd, kd, vd, od, ld, causal, scale, st, window, lens)

    if q.is_cuda:
        o = out if out is not None else torch.empty_like(q)
        ls = lse if lse is not None else torch.empty((B, H, N), dtype=torch.float32,
                                                     device=q.device)
        lens = None if seqlens_k is None else seqlens_k.to(q.device, torch.int32)
        run(q, k, v, o, ls, stream, lens)
        return o, ls
    dev = torch.device(device or "cuda:0")
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    o_host = out if out is not None else torch.empty(q.shape, dtype=q.dtype,
                                                     pin_memory=q.is_pinned())
    l_host = lse if lse is not None else torch.empty((B, H, N), dtype=torch.float32,
                                                     pin_memory=q.is_pinned())
    plain = (not split and all(t.is_contiguous() for t in (q, k, v, o_host, l_host))
             and q.dtype in (torch.bfloat16, torch.float16) and k.dtype == q.dtype
             and v.dtype == q.dtype and o_host.dtype == q.dtype)
    if plain:
        # fa_fwd_host_masked: the library copies group of heads by group of heads, overlapping
        # the copies of one group with the kernel of another.
        with torch.cuda.device(dev):
            qd, kd, vd, od = (torch.empty(q.shape, dtype=q.dtype, device=dev) for _ in range(4))
            ld = torch.empty((B, H, N), dtype=torch.float32, device=dev)
            lens = None if seqlens_k is None else seqlens_k.to(dev, torch.int32)
        left, right = (int(w) for w in window)
        rc = load_library().fa_fwd_host_masked(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o_host.data_ptr(), l_host.data_ptr(),
            qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(), ld.data_ptr(),
            B, H, N, d, int(bool(causal)), left, right,
            None if lens is None else lens.data_ptr(), float(scale), _dtype_code(q),
            st.cuda_stream)
        if rc != 0:
            raise FaError(rc, "fa_fwd_host_masked")
        st.synchronize()
        return o_host, l_host
    with torch.cuda.stream(st):
        qd, kd, vd = (t.to(dev, non_blocking=True) for t in (q, k, v))
        od = torch.empty_like(qd)
        ld = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        lens = None if seqlens_k is None else seqlens_k.to(dev, torch.int32, non_blocking=True)
        run(qd, kd, vd, od, ld, st, lens)
        o_host.copy_(od, non_blocking=True)
        l_host.copy_(ld, non_blocking=True)
    st.synchronize()
    return o_host, l_host


def attention_backward(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None,
                       stream=None, device=None, window=(-1, -1), seqlens_k=None):
    """dq, dk, dv = gradients of sum(dout * o) for o, lse = attention_forward(q, k, v, causal,
    window=window, seqlens_k=seqlens_k) (queries and keys share N).

    Device tensors are used in place; host tensors (ideally pinned) are copied to ``device``
    (default cuda:0), the kernels run there, and the gradients come back as host tensors.
    """
    import math

    import torch
    B, N, H, d = q.shape
    if scale is None:
        scale = float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))
    if q.is_cuda:
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        lens = None if seqlens_k is None else seqlens_k.to(q.device, torch.int32)
        fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, causal, scale, None, stream, window, lens)
        return dq, dk, dv
    for name, t in (("k", k), ("v", v), ("o", o), ("dout", dout)):
        if t.shape != q.shape or t.dtype != q.dtype or t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous host tensor like q" % name)
    if (q.dtype not in (torch.bfloat16, torch.float16) or not q.is_contiguous()
            or lse.shape != (B, H, N) or lse.dtype != torch.float32 or lse.is_cuda
            or not lse.is_contiguous()):
        raise ValueError("q must be a contiguous bf16/fp16 host tensor, lse float32 [B, H, N]")
    dev = torch.device(device or "cuda:0")
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    host = [torch.empty(q.shape, dtype=q.dtype, pin_memory=q.is_pinned()) for _ in range(3)]
    with torch.cuda.device(dev):
        bufs = [torch.empty(q.shape, dtype=q.dtype, device=dev) for _ in range(8)]
        ld = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        # 128 bytes beyond the whole problem's size: every head group gets a part of its own,
        # so that the groups' kernels overlap
        need = bwd_workspace_size(B, H, N, d) + 128
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        lens = None if seqlens_k is None else seqlens_k.to(dev, torch.int32)
    left, right = (int(w) for w in window)
    # fa_bwd_host_masked: copies of one group of heads overlap the kernels of another
    rc = load_library().fa_bwd_host_masked(
        *(t.data_ptr() for t in (q, k, v, o, dout, lse, *host)),
        *(t.data_ptr() for t in bufs[:5]), ld.data_ptr(), *(t.data_ptr() for t in bufs[5:]),
        ws.data_ptr(), need, B, H, N, d, int(bool(causal)), left, right,
        None if lens is None else lens.data_ptr(), float(scale), _dtype_code(q),
        st.cuda_stream)
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_host_masked")
    st.synchronize()
    return tuple(host)
