"""Python binding of libq4k.so, the GB300 Q4_K weight-matmul library.

Argument marshalling only: every function checks that its torch tensors are
contiguous CUDA tensors of the expected dtype, passes their device pointers
and the current torch stream to the C ABI (``include/q4k.h``) and raises
``Q4KError`` on a non-OK status.  All arithmetic runs in the library's CUDA
kernels; there is no CPU path.  Importing works without a GPU (the library
loads), but every compute call needs the CUDA device.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH, build

BLOCK144 = 0
LAYOUT_GPU = 1          # declared by the C ABI; every call refuses it (Q4K_ERR_UNSUPPORTED)
Q6K_GGUF = 0            # Q6_K 210-byte GGUF superblocks
Q6K_GPU = 1             # Q6_K GPU row layout (what q6k_gemv reads)
Q4K_OK = 0
QK_K = 256
QK_SUB = 32

_STATUS = {0: "Q4K_OK", 1: "Q4K_ERR_INVALID_ARG", 2: "Q4K_ERR_ALIGNMENT",
           3: "Q4K_ERR_UNSUPPORTED", 4: "Q4K_ERR_CUDA", 5: "Q4K_ERR_DEVICE_TIMEOUT"}

_P, _I64, _I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
GEMV_SEQ_MAX_JOBS = 256


class GemvJob(ctypes.Structure):
    """``q4k_gemv_job`` of the C ABI (one GEMV of a ``q4k_gemv_seq`` list)."""
    _fields_ = [("w", _P), ("rows", _I64), ("cols", _I64), ("x", _P), ("residual", _P), ("y", _P),
                ("wait", ctypes.c_int32), ("format", ctypes.c_int32)]


# Every symbol the header declares, with its ctypes signature.
SIGNATURES = {
    "q4k_packed_bytes": (ctypes.c_size_t, [_I64, _I64, _I]),
    "q4k_pack": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I, _P, _P]),
    "q4k_unpack": (_I, [_P, _I, _I64, _I64, _P, _P, _P, _P, _P, _P]),
    "q8_1_bytes": (ctypes.c_size_t, [_I64, _I64]),
    "q8_quantize": (_I, [_P, _I64, _I64, _P, _P, _P, _P]),
    "q8_quantize_h16": (_I, [_P, _I64, _I64, _P, _P, _P, _P]),
    "q4k_gemv": (_I, [_P, _I, _I64, _I64, _P, _I64, _P, _P, _P]),
    "q4k_gemv_q8": (_I, [_P, _I, _I64, _I64, _P, _P, _P, _I64, _P, _P, _P]),
    "q4k_gemv_multi": (_I, [_I, _P, _I, _P, _I64, _P, _I64, _P, _P, _P]),
    "q4k_gemv_seq_workspace_bytes": (ctypes.c_size_t, [_P, _I, _I64]),
    "q4k_gemv_seq": (_I, [_P, _I, _I, _I64, _P, ctypes.c_size_t, _P]),
    "q4k_gemv_seq_plan_bytes": (ctypes.c_size_t, [_I]),
    "q4k_gemv_seq_plan": (_I, [_P, _I, _I, _I64, _P, ctypes.c_size_t, _P, ctypes.c_size_t]),
    "q4k_gemv_seq_launch": (_I, [_P, _P]),
    "q4k_gemv_seq_launch_host": (_I, [_P, _P, _P, ctypes.c_size_t, _P, _P, ctypes.c_size_t, _P]),
    "q4k_gemv_seq_static": (_I, [_P, _I, _I, _I64, _P]),
    "q4k_gemm": (_I, [_P, _I, _I64, _I64, _P, _P, _P, _I64, _P, _P]),
    "q4k_gemm_blockdots": (_I, [_P, _I, _I64, _I64, _P, _I64, _P, _P]),
    "q4k_gemm_h16": (_I, [_P, _I, _I64, _I64, _P, _P, _P, _I64, _P, _P]),
    "q4k_gemm_blockdots_h16": (_I, [_P, _I, _I64, _I64, _P, _I64, _P, _P]),
    "x_split_f16_bytes": (ctypes.c_size_t, [_I64, _I64]),
    "x_split_f16": (_I, [_P, _I64, _I64, _P, _P, _P, _P, _P]),
    "q4k_gemm_f16": (_I, [_P, _I, _I64, _I64, _P, _P, _P, _P, _I64, _P, _P]),
    "q6k_packed_bytes": (ctypes.c_size_t, [_I64, _I64, _I]),
    "q6k_pack": (_I, [_P, _P, _P, _I64, _I64, _I, _P, _P]),
    "q6k_repack": (_I, [_P, _I, _I64, _I64, _P, _I, _P]),
    "q6k_unpack": (_I, [_P, _I, _I64, _I64, _P, _P, _P, _P]),
    "q6k_gemv": (_I, [_P, _I, _I64, _I64, _P, _I64, _P, _P, _P]),
    "q6k_gemv_q8": (_I, [_P, _I, _I64, _I64, _P, _P, _P, _I64, _P, _P, _P]),
    "q6k_gemm": (_I, [_P, _I, _I64, _I64, _P, _P, _P, _I64, _P, _P]),
    "q6k_gemm_blockdots": (_I, [_P, _I, _I64, _I64, _P, _I64, _P, _P]),
    "q6k_gemm_f16": (_I, [_P, _I, _I64, _I64, _P, _P, _P, _P, _I64, _P, _P]),
    "q4k_device_error": (_I, [_P]),
    "q4k_selftest_wait_timeout": (_I, [_P]),
    "q4k_status_string": (ctypes.c_char_p, [_I]),
    "q4k_last_error_string": (ctypes.c_char_p, []),
    "q4k_version": (ctypes.c_char_p, []),
}


class Q4KError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        detail = ""
        if status == 4 and _lib is not None:
            detail = ": " + _lib.q4k_last_error_string().decode()
        super().__init__(f"{call} failed with {_STATUS.get(status, status)}{detail}")


_lib = None


def lib() -> ctypes.CDLL:
    """Load libq4k.so (built in-tree by ``build()``); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run q4_weight_matmul_gb300.build.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t, dtype, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _ptr16(t, name):
    """binary16 bit patterns may arrive as uint16, int16 or float16 tensors."""
    kinds = (torch.int16, torch.float16) + ((torch.uint16,) if hasattr(torch, "uint16") else ())
    if not isinstance(t, torch.Tensor) or t.dtype not in kinds:
        raise TypeError(f"{name} must hold binary16 bits (uint16/int16/float16)")
    return _ptr(t, t.dtype, name)


def _check(status: int, call: str):
    if status != Q4K_OK:
        raise Q4KError(status, call)


def q4k_packed_bytes(rows: int, cols: int, layout: int = BLOCK144) -> int:
    return int(lib().q4k_packed_bytes(rows, cols, layout))


def q4k_pack(d, dmin, sc, m, q, out=None, layout: int = BLOCK144, stream=None):
    """Pack Q4_K fields (uint16 d/dmin bits, uint8 sc/m/q) into ``out``
    (uint8, ``q4k_packed_bytes`` long; allocated when None)."""
    rows, cols = q.shape
    if out is None:
        out = torch.empty(q4k_packed_bytes(rows, cols, layout), dtype=torch.uint8, device=q.device)
    _check(lib().q4k_pack(_ptr16(d, "d"), _ptr16(dmin, "dmin"),
                          _ptr(sc, torch.uint8, "sc"), _ptr(m, torch.uint8, "m"),
                          _ptr(q, torch.uint8, "q"), rows, cols, layout,
                          _ptr(out, torch.uint8, "out"), _stream(stream)), "q4k_pack")
    return out


def q4k_unpack(w, rows: int, cols: int, layout: int = BLOCK144, stream=None):
    """Test export: read the fields back out of packed weights; returns
    ``{"d", "dmin"}`` (int16 tensors holding binary16 bits) and ``{"sc", "m", "q"}`` (uint8)."""
    dev = w.device
    nb = cols // QK_K
    out = {"d": torch.empty((rows, nb), dtype=torch.int16, device=dev),
           "dmin": torch.empty((rows, nb), dtype=torch.int16, device=dev),
           "sc": torch.empty((rows, cols // QK_SUB), dtype=torch.uint8, device=dev),
           "m": torch.empty((rows, cols // QK_SUB), dtype=torch.uint8, device=dev),
           "q": torch.empty((rows, cols), dtype=torch.uint8, device=dev)}
    _check(lib().q4k_unpack(_ptr(w, torch.uint8, "w"), layout, rows, cols,
                            _ptr16(out["d"], "d"), _ptr16(out["dmin"], "dmin"),
                            _ptr(out["sc"], torch.uint8, "sc"), _ptr(out["m"], torch.uint8, "m"),
                            _ptr(out["q"], torch.uint8, "q"), _stream(stream)), "q4k_unpack")
    return out


def q8_1_bytes(tokens: int, cols: int) -> int:
    return int(lib().q8_1_bytes(tokens, cols))


def q8_quantize(x, q=None, d8=None, s=None, stream=None):
    """q8_1-quantise ``x`` [tokens][cols] float32; returns (q int8, d8 float32, sum int32)."""
    tokens, cols = x.shape
    dev = x.device
    q = torch.empty((tokens, cols), dtype=torch.int8, device=dev) if q is None else q
    d8 = torch.empty((tokens, cols // QK_SUB), dtype=torch.float32, device=dev) if d8 is None else d8
    s = torch.empty((tokens, cols // QK_SUB), dtype=torch.int32, device=dev) if s is None else s
    _check(lib().q8_quantize(_ptr(x, torch.float32, "x"), tokens, cols, _ptr(q, torch.int8, "q"),
                             _ptr(d8, torch.float32, "d8"), _ptr(s, torch.int32, "sum"),
                             _stream(stream)), "q8_quantize")
    return q, d8, s


def q8_quantize_h16(x, q=None, d8=None, s=None, stream=None):
    """q8_1-quantise ``x`` with the quants as binary16 (torch.float16 holding
    the integers -127..127); returns (q float16, d8 float32, sum int32)."""
    tokens, cols = x.shape
    dev = x.device
    q = torch.empty((tokens, cols), dtype=torch.float16, device=dev) if q is None else q
    d8 = torch.empty((tokens, cols // QK_SUB), dtype=torch.float32, device=dev) if d8 is None else d8
    s = torch.empty((tokens, cols // QK_SUB), dtype=torch.int32, device=dev) if s is None else s
    _check(lib().q8_quantize_h16(_ptr(x, torch.float32, "x"), tokens, cols, _ptr(q, torch.float16, "q"),
                                 _ptr(d8, torch.float32, "d8"), _ptr(s, torch.int32, "sum"),
                                 _stream(stream)), "q8_quantize_h16")
    return q, d8, s


def q4k_gemv(w, rows: int, cols: int, x, residual=None, y=None, layout: int = BLOCK144, stream=None):
    """Decode GEMV: ``y[b] = W x[b] (+ residual[b])`` for ``x`` [batch][cols] float32."""
    batch = x.shape[0]
    if y is None:
        y = torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    _check(lib().q4k_gemv(_ptr(w, torch.uint8, "w"), layout, rows, cols,
                          _ptr(x, torch.float32, "x"), batch,
                          _ptr(residual, torch.float32, "residual"),
                          _ptr(y, torch.float32, "y"), _stream(stream)), "q4k_gemv")
    return y


def q4k_gemv_q8(w, rows: int, cols: int, q8, d8, s, residual=None, y=None, layout: int = BLOCK144, stream=None):
    """MMQ GEMV over q8_1 activations (``q8_quantize`` output, 1..8 rows):
    ``y[b] = W x_hat[b] (+ residual[b])``."""
    batch = q8.shape[0]
    if y is None:
        y = torch.empty((batch, rows), dtype=torch.float32, device=q8.device)
    _check(lib().q4k_gemv_q8(_ptr(w, torch.uint8, "w"), layout, rows, cols, _ptr(q8, torch.int8, "q8"),
                             _ptr(d8, torch.float32, "d8"), _ptr(s, torch.int32, "sum"), batch,
                             _ptr(residual, torch.float32, "residual"), _ptr(y, torch.float32, "y"),
                             _stream(stream)), "q4k_gemv_q8")
    return y


def x_split_f16(x, out=None, stream=None):
    """Split ``x`` [tokens][cols] float32 for ``q4k_gemm_f16``: returns
    (hi, lo, bsum) as torch.float16 tensors and inv_scale float32 [tokens]."""
    tokens, cols = x.shape
    dev = x.device
    if out is None:
        out = (torch.empty((tokens, cols), dtype=torch.float16, device=dev),
               torch.empty((tokens, cols), dtype=torch.float16, device=dev),
               torch.empty((tokens, cols // QK_K, 16), dtype=torch.float16, device=dev),
               torch.empty((tokens,), dtype=torch.float32, device=dev))
    hi, lo, bs, inv = out
    _check(lib().x_split_f16(_ptr(x, torch.float32, "x"), tokens, cols, _ptr(hi, torch.float16, "hi"),
                             _ptr(lo, torch.float16, "lo"), _ptr(bs, torch.float16, "bsum"),
                             _ptr(inv, torch.float32, "inv_scale"), _stream(stream)), "x_split_f16")
    return out


def q4k_gemm_f16(w, rows: int, cols: int, hi, lo, bsum, inv_scale, y=None, layout: int = BLOCK144, stream=None):
    """fp16-activation prefill GEMM over ``x_split_f16`` output: ``y = x W^T``."""
    tokens = hi.shape[0]
    if y is None:
        y = torch.empty((tokens, rows), dtype=torch.float32, device=hi.device)
    _check(lib().q4k_gemm_f16(_ptr(w, torch.uint8, "w"), layout, rows, cols, _ptr(hi, torch.float16, "hi"),
                              _ptr(lo, torch.float16, "lo"), _ptr(bsum, torch.float16, "bsum"),
                              _ptr(inv_scale, torch.float32, "inv_scale"), tokens, _ptr(y, torch.float32, "y"),
                              _stream(stream)), "q4k_gemm_f16")
    return y


def q6k_packed_bytes(rows: int, cols: int, layout: int = Q6K_GPU) -> int:
    return int(lib().q6k_packed_bytes(rows, cols, layout))


def q6k_pack(d, sc, q, out=None, layout: int = Q6K_GPU, stream=None):
    """Pack Q6_K fields (binary16 d bits [rows][cols/256], int8 sc
    [rows][cols/16], uint8 q [rows][cols]) into ``out`` (uint8,
    ``q6k_packed_bytes`` long; allocated when None)."""
    rows, cols = q.shape
    if out is None:
        out = torch.empty(q6k_packed_bytes(rows, cols, layout), dtype=torch.uint8, device=q.device)
    _check(lib().q6k_pack(_ptr16(d, "d"), _ptr(sc, torch.int8, "sc"), _ptr(q, torch.uint8, "q"), rows, cols,
                          layout, _ptr(out, torch.uint8, "out"), _stream(stream)), "q6k_pack")
    return out


def q6k_repack(src, rows: int, cols: int, src_layout: int = Q6K_GGUF, dst_layout: int = Q6K_GPU, out=None,
               stream=None):
    """Convert packed Q6_K weights between layouts (GGUF blocks to the GPU layout by default)."""
    if out is None:
        out = torch.empty(q6k_packed_bytes(rows, cols, dst_layout), dtype=torch.uint8, device=src.device)
    _check(lib().q6k_repack(_ptr(src, torch.uint8, "src"), src_layout, rows, cols,
                            _ptr(out, torch.uint8, "out"), dst_layout, _stream(stream)), "q6k_repack")
    return out


def q6k_unpack(w, rows: int, cols: int, layout: int = Q6K_GPU, stream=None):
    """Test export: the fields of packed Q6_K weights, ``{"d"}`` (int16
    binary16 bits), ``{"sc"}`` (int8) and ``{"q"}`` (uint8)."""
    dev = w.device
    out = {"d": torch.empty((rows, cols // QK_K), dtype=torch.int16, device=dev),
           "sc": torch.empty((rows, cols // 16), dtype=torch.int8, device=dev),
           "q": torch.empty((rows, cols), dtype=torch.uint8, device=dev)}
    _check(lib().q6k_unpack(_ptr(w, torch.uint8, "w"), layout, rows, cols, _ptr16(out["d"], "d"),
                            _ptr(out["sc"], torch.int8, "sc"), _ptr(out["q"], torch.uint8, "q"),
                            _stream(stream)), "q6k_unpack")
    return out


def q6k_gemv(w, rows: int, cols: int, x, residual=None, y=None, layout: int = Q6K_GPU, stream=None):
    """Decode GEMV over Q6_K weights (GPU layout): ``y[b] = W x[b] (+ residual[b])``."""
    batch = x.shape[0]
    if y is None:
        y = torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    _check(lib().q6k_gemv(_ptr(w, torch.uint8, "w"), layout, rows, cols, _ptr(x, torch.float32, "x"), batch,
                          _ptr(residual, torch.float32, "residual"), _ptr(y, torch.float32, "y"),
                          _stream(stream)), "q6k_gemv")
    return y


def q6k_gemv_q8(w, rows: int, cols: int, q8, d8, s=None, residual=None, y=None, layout: int = Q6K_GPU, stream=None):
    """MMQ GEMV over Q6_K weights and q8_1 activations (1..8 rows)."""
    batch = q8.shape[0]
    if y is None:
        y = torch.empty((batch, rows), dtype=torch.float32, device=q8.device)
    _check(lib().q6k_gemv_q8(_ptr(w, torch.uint8, "w"), layout, rows, cols, _ptr(q8, torch.int8, "q8"),
                             _ptr(d8, torch.float32, "d8"), _ptr(s, torch.int32, "sum"), batch,
                             _ptr(residual, torch.float32, "residual"), _ptr(y, torch.float32, "y"),
                             _stream(stream)), "q6k_gemv_q8")
    return y


def q6k_gemm(w, rows: int, cols: int, q8, d8, s=None, y=None, layout: int = Q6K_GPU, stream=None):
    """MMQ product over Q6_K weights for any number of q8_1 token rows."""
    tokens = q8.shape[0]
    if y is None:
        y = torch.empty((tokens, rows), dtype=torch.float32, device=q8.device)
    _check(lib().q6k_gemm(_ptr(w, torch.uint8, "w"), layout, rows, cols, _ptr(q8, torch.int8, "q8"),
                          _ptr(d8, torch.float32, "d8"), _ptr(s, torch.int32, "sum"), tokens,
                          _ptr(y, torch.float32, "y"), _stream(stream)), "q6k_gemm")
    return y


def q6k_gemm_f16(w, rows: int, cols: int, hi, lo, bsum, inv_scale, y=None, layout: int = Q6K_GPU, stream=None):
    """fp16-activation tensor-core GEMM over Q6_K weights, on ``x_split_f16`` output."""
    tokens = hi.shape[0]
    if y is None:
        y = torch.empty((tokens, rows), dtype=torch.float32, device=hi.device)
    bs = None if bsum is None else _ptr(bsum, torch.float16, "bsum")
    _check(lib().q6k_gemm_f16(_ptr(w, torch.uint8, "w"), layout, rows, cols, _ptr(hi, torch.float16, "hi"),
                              _ptr(lo, torch.float16, "lo"), bs, _ptr(inv_scale, torch.float32, "inv_scale"),
                              tokens, _ptr(y, torch.float32, "y"), _stream(stream)), "q6k_gemm_f16")
    return y


def q6k_gemm_blockdots(w, rows: int, cols: int, q8, layout: int = Q6K_GPU, stream=None):
    """Test export: the exact 16-weight group dots [tokens][rows][cols/16] (int32)."""
    tokens = q8.shape[0]
    p = torch.empty((tokens, rows, cols // 16), dtype=torch.int32, device=q8.device)
    _check(lib().q6k_gemm_blockdots(_ptr(w, torch.uint8, "w"), layout, rows, cols, _ptr(q8, torch.int8, "q8"),
                                    tokens, _ptr(p, torch.int32, "p"), _stream(stream)), "q6k_gemm_blockdots")
    return p


def q4k_gemv_multi(ws, rows, cols: int, x, residuals=None, ys=None, layout: int = BLOCK144, stream=None):
    """One launch of several GEMVs sharing ``x``: ``ys[m] = W_m x (+ residuals[m])``."""
    n = len(ws)
    batch = x.shape[0]
    if ys is None:
        ys = [torch.empty((batch, r), dtype=torch.float32, device=x.device) for r in rows]
    wp = (ctypes.c_void_p * n)(*[_ptr(w, torch.uint8, "w") for w in ws])
    rp = (ctypes.c_int64 * n)(*[int(r) for r in rows])
    yp = (ctypes.c_void_p * n)(*[_ptr(y, torch.float32, "y") for y in ys])
    resp = None
    if residuals is not None:
        resp = (ctypes.c_void_p * n)(*[_ptr(r, torch.float32, "residual") for r in residuals])
    _check(lib().q4k_gemv_multi(n, wp, layout, rp, cols, _ptr(x, torch.float32, "x"), batch,
                                resp, yp, _stream(stream)), "q4k_gemv_multi")
    return ys


def _job_array(jobs):
    n = len(jobs)
    arr = (GemvJob * max(n, 1))()
    dev = None
    for i, j in enumerate(jobs):
        arr[i].w = _ptr(j["w"], torch.uint8, "w")
        arr[i].rows = int(j["rows"])
        arr[i].cols = int(j["cols"])
        arr[i].x = _ptr(j["x"], torch.float32, "x")
        arr[i].residual = _ptr(j.get("residual"), torch.float32, "residual")
        arr[i].y = _ptr(j["y"], torch.float32, "y")
        arr[i].wait = 1 if j.get("wait") else 0
        arr[i].format = int(j.get("format", 0))      # 0 Q4_K, 1 Q6_K (GPU layout)
        dev = j["x"].device if dev is None else dev
    return arr, n, dev


def _workspace(arr, n, batch, dev, workspace):
    need = int(lib().q4k_gemv_seq_workspace_bytes(arr, n, batch)) if n else 0
    if workspace is None:
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev)
    elif workspace.numel() < need:
        raise ValueError(f"workspace holds {workspace.numel()} bytes, the job list needs {need}")
    return workspace, need


class GemvSeq:
    """A prepared ``q4k_gemv_seq`` job list: the C job array, a zeroed
    workspace and the host plan (``q4k_gemv_seq_plan``), built once; calling
    it enqueues the plan's persistent launch (``q4k_gemv_seq_launch``).

    ``jobs`` is a sequence of dicts with keys ``w`` (packed uint8), ``rows``,
    ``cols``, ``x`` ([batch][cols] float32), ``y`` ([batch][rows] float32),
    optional ``residual`` and ``wait`` (read x only after every earlier job
    has stored its y).  The tensors must stay alive while the list is used.
    """

    def __init__(self, jobs, batch: int, layout: int = BLOCK144, workspace=None):
        arr, n, dev = _job_array(jobs)
        self.jobs, self.n, self.batch, self.layout = arr, n, int(batch), layout
        self.workspace, self.workspace_bytes = _workspace(arr, n, self.batch, dev, workspace)
        nbytes = int(lib().q4k_gemv_seq_plan_bytes(n))
        if nbytes == 0:
            raise Q4KError(3, "q4k_gemv_seq_plan_bytes")
        self._plan_buf = ctypes.create_string_buffer(nbytes + 64)
        base = ctypes.addressof(self._plan_buf)
        self.plan = base + (-base) % 64          # the plan must be 64-byte aligned
        _check(lib().q4k_gemv_seq_plan(arr, n, layout, self.batch,
                                       _ptr(self.workspace, torch.uint8, "workspace"),
                                       self.workspace.numel(), self.plan, nbytes), "q4k_gemv_seq_plan")

    def __call__(self, stream=None):
        _check(lib().q4k_gemv_seq_launch(self.plan, _stream(stream)), "q4k_gemv_seq_launch")

    def launch_host(self, x_host, x_dev, y_host, y_dev, stream=None):
        """One step from host buffers (``q4k_gemv_seq_launch_host``): copy
        ``x_host`` into ``x_dev``, launch, copy ``y_dev`` into ``y_host``, all
        enqueued on the stream.  The jobs' x and y must be views of ``x_dev``
        and ``y_dev``; the host tensors should be pinned.  Synchronise the
        stream before reading ``y_host``."""
        def _host(t, name):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous host tensor")
            return t.data_ptr(), t.numel() * t.element_size()

        def _dev(t, name, nbytes):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous device tensor")
            if t.numel() * t.element_size() < nbytes:
                raise ValueError(f"{name} is smaller than its host buffer")
            return t.data_ptr()

        xh, xb = _host(x_host, "x_host")
        yh, yb = _host(y_host, "y_host")
        _check(lib().q4k_gemv_seq_launch_host(self.plan, xh, _dev(x_dev, "x_dev", xb), xb, yh,
                                              _dev(y_dev, "y_dev", yb), yb, _stream(stream)),
               "q4k_gemv_seq_launch_host")

    def bind_host(self, x_host, x_dev, y_host, y_dev):
        """Check the four buffers of ``launch_host`` once and keep them (and
        references to them), so that ``step`` passes only pointers."""
        for t, name, cuda in ((x_host, "x_host", False), (x_dev, "x_dev", True), (y_host, "y_host", False),
                              (y_dev, "y_dev", True)):
            if t.is_cuda != cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous {'device' if cuda else 'host'} tensor")
        xb, yb = x_host.numel() * x_host.element_size(), y_host.numel() * y_host.element_size()
        if x_dev.numel() * x_dev.element_size() < xb or y_dev.numel() * y_dev.element_size() < yb:
            raise ValueError("a device buffer is smaller than its host buffer")
        self._bound = (x_host, x_dev, y_host, y_dev)
        self._bound_args = (x_host.data_ptr(), x_dev.data_ptr(), xb, y_host.data_ptr(), y_dev.data_ptr(), yb)

    def step(self, stream=None):
        """``launch_host`` on the buffers given to ``bind_host``."""
        xh, xd, xb, yh, yd, yb = self._bound_args
        _check(lib().q4k_gemv_seq_launch_host(self.plan, xh, xd, xb, yh, yd, yb, _stream(stream)),
               "q4k_gemv_seq_launch_host")


def q4k_gemv_seq(jobs, batch: int, layout: int = BLOCK144, workspace=None, stream=None):
    """One call of ``q4k_gemv_seq`` (plan and launch in one) over an ordered
    GEMV job list (see ``GemvSeq``); returns the workspace it used."""
    arr, n, dev = _job_array(jobs)
    workspace, _ = _workspace(arr, n, int(batch), dev, workspace)
    _check(lib().q4k_gemv_seq(arr, n, layout, int(batch), _ptr(workspace, torch.uint8, "workspace"),
                              workspace.numel(), _stream(stream)), "q4k_gemv_seq")
    return workspace


def q4k_gemv_seq_static(jobs, batch: int, layout: int = BLOCK144, stream=None):
    """``q4k_gemv_seq`` without a workspace: the library's built-in scratch
    array serves instead, so nothing is allocated (for callers that cannot
    allocate device memory).  Calls that overlap on the GPU race."""
    arr, n, _ = _job_array(jobs)
    _check(lib().q4k_gemv_seq_static(arr, n, layout, int(batch), _stream(stream)), "q4k_gemv_seq_static")


def q4k_gemm(w, rows: int, cols: int, q8, d8, s, y=None, layout: int = BLOCK144, stream=None):
    """Prefill MMQ GEMM on q8_1 activations; returns ``y`` [tokens][rows] float32."""
    tokens = q8.shape[0]
    if y is None:
        y = torch.empty((tokens, rows), dtype=torch.float32, device=q8.device)
    _check(lib().q4k_gemm(_ptr(w, torch.uint8, "w"), layout, rows, cols,
                          _ptr(q8, torch.int8, "q8"), _ptr(d8, torch.float32, "d8"),
                          _ptr(s, torch.int32, "sum"), tokens, _ptr(y, torch.float32, "y"),
                          _stream(stream)), "q4k_gemm")
    return y


def q4k_gemm_h16(w, rows: int, cols: int, q16, d8, s, y=None, layout: int = BLOCK144, stream=None):
    """Prefill MMQ GEMM on ``q8_quantize_h16`` output; returns ``y`` [tokens][rows] float32."""
    tokens = q16.shape[0]
    if y is None:
        y = torch.empty((tokens, rows), dtype=torch.float32, device=q16.device)
    _check(lib().q4k_gemm_h16(_ptr(w, torch.uint8, "w"), layout, rows, cols,
                              _ptr(q16, torch.float16, "q16"), _ptr(d8, torch.float32, "d8"),
                              _ptr(s, torch.int32, "sum"), tokens, _ptr(y, torch.float32, "y"),
                              _stream(stream)), "q4k_gemm_h16")
    return y


def q4k_gemm_blockdots_h16(w, rows: int, cols: int, q16, p=None, layout: int = BLOCK144, stream=None):
    """Test export: q4k_gemm_h16's exact per-block integer dots, int32 [tokens][rows][cols/32]."""
    tokens = q16.shape[0]
    if p is None:
        p = torch.empty((tokens, rows, cols // QK_SUB), dtype=torch.int32, device=q16.device)
    _check(lib().q4k_gemm_blockdots_h16(_ptr(w, torch.uint8, "w"), layout, rows, cols,
                                        _ptr(q16, torch.float16, "q16"), tokens,
                                        _ptr(p, torch.int32, "p"), _stream(stream)),
           "q4k_gemm_blockdots_h16")
    return p


def q4k_gemm_blockdots(w, rows: int, cols: int, q8, p=None, layout: int = BLOCK144, stream=None):
    """Test export: the GEMM's exact per-block integer dots, int32 [tokens][rows][cols/32]."""
    tokens = q8.shape[0]
    if p is None:
        p = torch.empty((tokens, rows, cols // QK_SUB), dtype=torch.int32, device=q8.device)
    _check(lib().q4k_gemm_blockdots(_ptr(w, torch.uint8, "w"), layout, rows, cols,
                                    _ptr(q8, torch.int8, "q8"), tokens,
                                    _ptr(p, torch.int32, "p"), _stream(stream)),
           "q4k_gemm_blockdots")
    return p


def q4k_device_error(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device error status."""
    return int(lib().q4k_device_error(_stream(stream)))


def q4k_selftest_wait_timeout(stream=None) -> None:
    """Enqueue the library's bounded-wait self-test kernel (see q4k.h); the
    next ``q4k_device_error`` reports the timeout it records."""
    _check(lib().q4k_selftest_wait_timeout(_stream(stream)), "q4k_selftest_wait_timeout")


def q4k_version() -> str:
    return lib().q4k_version().decode()


__all__ = ["build", "lib", "Q4KError", "BLOCK144", "LAYOUT_GPU", "q4k_packed_bytes", "q4k_pack", "q4k_unpack",
           "q4k_gemv_q8",
           "q8_1_bytes", "q8_quantize", "q8_quantize_h16", "q4k_gemm_h16", "q4k_gemm_blockdots_h16",
           "q4k_gemv", "q4k_gemv_multi", "GemvJob", "GemvSeq", "q4k_gemv_seq", "q4k_gemv_seq_static", "q4k_gemm",
           "q4k_gemm_blockdots", "q4k_device_error",
           "q4k_selftest_wait_timeout", "q4k_version",
           "SIGNATURES"]
