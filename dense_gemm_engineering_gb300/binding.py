"""Python binding of the C ABI in include/gemm.h (argument marshalling only).

Every function here forwards to libgb300gemm.so through ctypes: it reads data
pointers, strides and the current CUDA stream from torch tensors and passes
them on.  No arithmetic of the GEMM runs in Python and there is no fallback:
if the library is missing or the call fails, a GemmError is raised.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

GEMM_F16, GEMM_BF16, GEMM_E4M3, GEMM_E5M2 = 0, 1, 2, 3
LAYOUT_ABT, LAYOUT_AB = 0, 1

STATUS_NAMES = {
    0: "GEMM_OK",
    -1: "GEMM_ERR_NULL",
    -2: "GEMM_ERR_DTYPE",
    -3: "GEMM_ERR_SHAPE",
    -4: "GEMM_ERR_ALIGN",
    -5: "GEMM_ERR_ALIAS",
    -6: "GEMM_ERR_CUDA",
    -7: "GEMM_ERR_DEVICE",
    -8: "GEMM_ERR_OPTION",
    -9: "GEMM_ERR_TIMEOUT",
    -10: "GEMM_ERR_WORKSPACE",
}

# Every symbol include/gemm.h declares.
EXPORTS = ("gemm_abt", "gemm_ab", "gemm_run", "gemm_run_workspace", "gemm_workspace_size",
           "gemm_run_no_alloc", "gemm_status_string", "gemm_plan", "gemm_tile_origin",
           "gemm_device_status", "gemm_selftest_wait_timeout", "gemm_selftest_gemm_timeout",
           "gemm_run_clock_probe",
           "gemm_fp8_abt", "gemm_fp8_run",
           "gemm_fp8_run_workspace", "gemm_mx_abt", "gemm_mx_run", "gemm_mx_scales_size",
           "gemm_mx_scales_b_size", "gemm_mx_pack_scales", "gemm_mx_pack_scales_b", "gemm_mx_plan")


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = f"{STATUS_NAMES.get(status, status)}: {gemm_status_string(status)}"
        super().__init__(f"{what}: {msg}" if what else msg)


class GemmOptions(ctypes.Structure):
    """gemm_options_t."""
    _fields_ = [("cta_group", ctypes.c_int), ("block_n", ctypes.c_int),
                ("raster_group", ctypes.c_int), ("max_clusters", ctypes.c_int),
                ("tail_split", ctypes.c_int), ("consumers", ctypes.c_int),
                ("multicast", ctypes.c_int), ("raster_order", ctypes.c_int),
                ("l2_hints", ctypes.c_int), ("cluster_ksplit", ctypes.c_int)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load the CUDA library (built in-tree by build.build())."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(
            f"CUDA library {p} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    vp, i64, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    ip = ctypes.POINTER(c_int)
    for name in ("gemm_abt", "gemm_ab"):
        f = getattr(lib, name)
        f.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int, vp]
        f.restype = c_int
    lib.gemm_run.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int, c_int,
                             ctypes.POINTER(GemmOptions), vp]
    lib.gemm_run.restype = c_int
    lib.gemm_run_workspace.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int, c_int,
                                       ctypes.POINTER(GemmOptions), vp, ctypes.c_size_t, vp]
    lib.gemm_run_workspace.restype = c_int
    lib.gemm_workspace_size.argtypes = [i64, i64, i64, c_int, c_int, ctypes.POINTER(GemmOptions),
                                        ctypes.POINTER(ctypes.c_size_t)]
    lib.gemm_workspace_size.restype = c_int
    lib.gemm_run_no_alloc.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int, c_int,
                                      ctypes.POINTER(GemmOptions), vp]
    lib.gemm_run_no_alloc.restype = c_int
    f32 = ctypes.c_float
    lib.gemm_fp8_abt.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int, c_int, f32, vp]
    lib.gemm_fp8_abt.restype = c_int
    lib.gemm_fp8_run.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int, c_int, f32,
                                 ctypes.POINTER(GemmOptions), vp]
    lib.gemm_fp8_run.restype = c_int
    lib.gemm_fp8_run_workspace.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int, c_int,
                                           f32, ctypes.POINTER(GemmOptions), vp, ctypes.c_size_t, vp]
    lib.gemm_fp8_run_workspace.restype = c_int
    lib.gemm_mx_abt.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int, c_int,
                                f32, vp]
    lib.gemm_mx_abt.restype = c_int
    lib.gemm_mx_run.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int, c_int,
                                f32, ctypes.POINTER(GemmOptions), vp]
    lib.gemm_mx_run.restype = c_int
    lib.gemm_mx_scales_size.argtypes = [i64, i64, ctypes.POINTER(ctypes.c_size_t)]
    lib.gemm_mx_scales_size.restype = c_int
    lib.gemm_mx_scales_b_size.argtypes = [i64, i64, ctypes.POINTER(ctypes.c_size_t)]
    lib.gemm_mx_scales_b_size.restype = c_int
    lib.gemm_mx_pack_scales.argtypes = [vp, i64, i64, i64, vp, vp]
    lib.gemm_mx_pack_scales.restype = c_int
    lib.gemm_mx_pack_scales_b.argtypes = [vp, i64, i64, i64, vp, vp]
    lib.gemm_mx_pack_scales_b.restype = c_int
    lib.gemm_mx_plan.argtypes = [i64, i64, i64, c_int, ctypes.POINTER(GemmOptions), ip, ip, ip,
                                 ip, ip, ctypes.POINTER(i64), ip, ip]
    lib.gemm_mx_plan.restype = c_int
    lib.gemm_status_string.argtypes = [c_int]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_plan.argtypes = [i64, i64, i64, c_int, c_int, ctypes.POINTER(GemmOptions), ip, ip,
                              ip, ip, ip, ctypes.POINTER(i64), ip, ip, ip, ip, ip]
    lib.gemm_plan.restype = c_int
    lib.gemm_tile_origin.argtypes = [i64, i64, c_int, c_int, c_int, c_int, i64, ctypes.POINTER(i64),
                                     ctypes.POINTER(i64)]
    lib.gemm_tile_origin.restype = c_int
    lib.gemm_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), c_int]
    lib.gemm_device_status.restype = c_int
    lib.gemm_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    lib.gemm_selftest_wait_timeout.restype = c_int
    lib.gemm_selftest_gemm_timeout.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int,
                                               c_int, ctypes.POINTER(GemmOptions),
                                               ctypes.c_uint64, vp]
    lib.gemm_selftest_gemm_timeout.restype = c_int
    lib.gemm_run_clock_probe.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int, c_int,
                                         ctypes.POINTER(GemmOptions), vp, vp]
    lib.gemm_run_clock_probe.restype = c_int
    if path is None:
        _lib = lib
    return lib


def gemm_status_string(status: int) -> str:
    return load().gemm_status_string(int(status)).decode()


_options_cache = {}


def _options_key(options):
    if options is None:
        return None
    if isinstance(options, GemmOptions):
        return tuple(getattr(options, f) for f, _ in GemmOptions._fields_)
    return tuple(sorted((k, int(v)) for k, v in dict(options).items()))


def _options(options) -> ctypes.POINTER(GemmOptions) | None:
    if options is None:
        return None
    if isinstance(options, GemmOptions):
        return ctypes.pointer(options)
    key = _options_key(options)
    p = _options_cache.get(key)
    if p is None:
        p = ctypes.pointer(GemmOptions(**dict(key)))
        _options_cache[key] = p
    return p


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.float16:
        return GEMM_F16
    if t.dtype == torch.bfloat16:
        return GEMM_BF16
    raise GemmError(-2, f"tensor dtype {t.dtype}")


def _ld(t, multiple: int = 8) -> int:
    # Row stride in elements of a row-major 2-D view (inner stride must be 1).
    if t.dim() != 2:
        raise GemmError(-3, "operands must be 2-D")
    if t.shape[0] > 0 and t.shape[1] > 1 and t.stride(1) != 1:
        raise GemmError(-3, "inner dimension must be contiguous")
    if t.shape[0] > 1:
        return int(t.stride(0))
    # one row (or none): the stride is never used; any legal value will do
    m = multiple
    return max(m, (int(t.shape[1]) + m - 1) // m * m)


def _fp8_code(t, fmt) -> int:
    """GEMM_E4M3 / GEMM_E5M2 for a torch float8 tensor, or for a uint8 tensor of
    FP8 bit patterns with `fmt` = "e4m3" / "e5m2"."""
    import torch

    by_dtype = {getattr(torch, "float8_e4m3fn", None): GEMM_E4M3,
                getattr(torch, "float8_e5m2", None): GEMM_E5M2}
    if t.dtype in by_dtype and t.dtype is not None:
        code = by_dtype[t.dtype]
        if fmt is not None and {"e4m3": GEMM_E4M3, "e5m2": GEMM_E5M2}.get(fmt) != code:
            raise GemmError(-2, f"fmt {fmt!r} does not match tensor dtype {t.dtype}")
        return code
    if t.dtype == torch.uint8 and fmt in ("e4m3", "e5m2"):
        return GEMM_E4M3 if fmt == "e4m3" else GEMM_E5M2
    raise GemmError(-2, f"FP8 operands: float8 tensors, or uint8 with fmt='e4m3'/'e5m2' "
                        f"(got {t.dtype}, fmt={fmt!r})")


def _stream_handle(stream, device) -> int:
    import torch

    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


# Workspaces for the split tail, one per (device, stream): calls on one stream
# run in order, so they may share one; calls on different streams must not.
_workspaces = {}
# gemm_workspace_size results per (shape, dtype, layout, options, device).
_ws_need_cache = {}


def _workspace(device, stream_handle: int, nbytes: int):
    import torch

    key = (device.index if device.index is not None else torch.cuda.current_device(),
           stream_handle)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        # zeroed once when (re)allocated, as gemm_run_workspace requires
        ws = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def gemm_run(A, B, D=None, *, layout: int = LAYOUT_ABT, options=None, stream=None,
             workspace="auto"):
    """D = A.B^T (layout 0, B is N x K) or A.B (layout 1, B is K x N) on torch tensors.

    Allocates D with torch when not given.  Enqueues on `stream` (default: the
    current stream of A's device) and returns D without synchronising.
    `workspace`: "auto" (a zero-initialised device buffer kept per device and
    stream, sized by gemm_workspace_size), None (no workspace: the plain
    persistent schedule), or a caller-owned uint8 CUDA tensor.
    """
    import torch

    if A.device.type != "cuda" or B.device.type != "cuda":
        raise GemmError(-1, "operands must be CUDA tensors")
    M, K = A.shape
    N = B.shape[0] if layout == LAYOUT_ABT else B.shape[1]
    Kb = B.shape[1] if layout == LAYOUT_ABT else B.shape[0]
    if Kb != K:
        raise GemmError(-3, f"K mismatch ({K} vs {Kb})")
    if A.dtype != B.dtype:
        raise GemmError(-2, "A and B must share a dtype")
    if D is None:
        D = torch.empty((M, N), dtype=A.dtype, device=A.device)
    elif D.dtype != A.dtype or tuple(D.shape) != (M, N):
        raise GemmError(-3, "D has the wrong dtype or shape")
    lib = load()
    sh = _stream_handle(stream, A.device)
    opts = _options(options)
    dt = _dtype_code(A)
    ws_ptr, ws_bytes = None, 0
    if isinstance(workspace, str) and workspace == "auto":
        dev_index = A.device.index if A.device.index is not None else torch.cuda.current_device()
        key = (M, N, K, dt, int(layout), _options_key(options), dev_index)
        need = _ws_need_cache.get(key)
        if need is None:
            n = ctypes.c_size_t()
            st = lib.gemm_workspace_size(M, N, K, dt, int(layout), opts, ctypes.byref(n))
            if st != 0:
                raise GemmError(st, "gemm_workspace_size")
            need = _ws_need_cache[key] = n.value
        if need:
            ws = _workspace(A.device, sh, need)
            ws_ptr, ws_bytes = ws.data_ptr(), ws.numel()
    elif workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = lib.gemm_run_workspace(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, _ld(A),
                                _ld(B), _ld(D), dt, int(layout), opts, ws_ptr, ws_bytes, sh)
    if st != 0:
        raise GemmError(st, "gemm_run_workspace")
    return D


def gemm_fp8(A, B, D=None, *, fmt=None, out_dtype=None, alpha: float = 1.0, options=None,
             stream=None, workspace="auto"):
    """D[M, N] = alpha * A[M, K] . B[N, K]^T with FP8 A and B (both E4M3 or both
    E5M2: torch float8 tensors, or uint8 bit patterns with `fmt`), FP32
    accumulation and a 16-bit D (`out_dtype`, default bfloat16)."""
    import torch

    if A.device.type != "cuda" or B.device.type != "cuda":
        raise GemmError(-1, "operands must be CUDA tensors")
    code = _fp8_code(A, fmt)
    if _fp8_code(B, fmt) != code:
        raise GemmError(-2, "A and B must share an FP8 format")
    M, K = A.shape
    N, Kb = B.shape
    if Kb != K:
        raise GemmError(-3, f"K mismatch ({K} vs {Kb})")
    odt = out_dtype if out_dtype is not None else (D.dtype if D is not None else torch.bfloat16)
    if D is None:
        D = torch.empty((M, N), dtype=odt, device=A.device)
    elif D.dtype != odt or tuple(D.shape) != (M, N):
        raise GemmError(-3, "D has the wrong dtype or shape")
    out_code = _dtype_code(D)
    lib = load()
    sh = _stream_handle(stream, A.device)
    opts = _options(options)
    ws_ptr, ws_bytes = None, 0
    if isinstance(workspace, str) and workspace == "auto":
        dev_index = A.device.index if A.device.index is not None else torch.cuda.current_device()
        key = (M, N, K, code, LAYOUT_ABT, _options_key(options), dev_index)
        need = _ws_need_cache.get(key)
        if need is None:
            n = ctypes.c_size_t()
            st = lib.gemm_workspace_size(M, N, K, code, LAYOUT_ABT, opts, ctypes.byref(n))
            if st != 0:
                raise GemmError(st, "gemm_workspace_size")
            need = _ws_need_cache[key] = n.value
        if need:
            ws = _workspace(A.device, sh, need)
            ws_ptr, ws_bytes = ws.data_ptr(), ws.numel()
    elif workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = lib.gemm_fp8_run_workspace(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                                    _ld(A, 16), _ld(B, 16), _ld(D), code, out_code, float(alpha),
                                    opts, ws_ptr, ws_bytes, sh)
    if st != 0:
        raise GemmError(st, "gemm_fp8_run_workspace")
    return D


def gemm_abt(A, B, D=None, *, options=None, stream=None, workspace="auto"):
    """D[M, N] = A[M, K] . B[N, K]^T (FP16/BF16, FP32 accumulation)."""
    return gemm_run(A, B, D, layout=LAYOUT_ABT, options=options, stream=stream,
                    workspace=workspace)


def gemm_ab(A, B, D=None, *, options=None, stream=None, workspace="auto"):
    """D[M, N] = A[M, K] . B[K, N] (FP16/BF16, FP32 accumulation)."""
    return gemm_run(A, B, D, layout=LAYOUT_AB, options=options, stream=stream,
                    workspace=workspace)


def gemm_workspace_size(M: int, N: int, K: int, dtype: int = GEMM_F16,
                        layout: int = LAYOUT_ABT, options=None) -> int:
    """Bytes of workspace the split tail needs on the current device (0 = none)."""
    need = ctypes.c_size_t()
    st = load().gemm_workspace_size(M, N, K, dtype, layout, _options(options),
                                    ctypes.byref(need))
    if st != 0:
        raise GemmError(st, "gemm_workspace_size")
    return need.value


def gemm_run_ptr(A: int, B: int, D: int, M: int, N: int, K: int, lda: int, ldb: int, ldd: int,
                 dtype: int, layout: int = LAYOUT_ABT, options=None, stream: int = 0,
                 workspace: int = 0, workspace_bytes: int = 0) -> int:
    """The raw C call on integer addresses; returns the status code."""
    if workspace:
        return load().gemm_run_workspace(A, B, D, M, N, K, lda, ldb, ldd, dtype, layout,
                                         _options(options), workspace, workspace_bytes, stream)
    return load().gemm_run(A, B, D, M, N, K, lda, ldb, ldd, dtype, layout, _options(options),
                           stream)


def mx_scales_size(rows: int, K: int) -> int:
    """Bytes of the block scales of A (rows = M) in the layout gemm_mx reads."""
    n = ctypes.c_size_t()
    st = load().gemm_mx_scales_size(int(rows), int(K), ctypes.byref(n))
    if st != 0:
        raise GemmError(st, "gemm_mx_scales_size")
    return n.value


def mx_scales_b_size(N: int, K: int) -> int:
    """Bytes of the block scales of B in the layout gemm_mx reads."""
    n = ctypes.c_size_t()
    st = load().gemm_mx_scales_b_size(int(N), int(K), ctypes.byref(n))
    if st != 0:
        raise GemmError(st, "gemm_mx_scales_b_size")
    return n.value


def _pack(S, K, out, stream, for_b):
    import torch

    if S.device.type != "cuda" or S.dtype != torch.uint8 or S.dim() != 2:
        raise GemmError(-2, "scales: a 2-D uint8 CUDA tensor")
    rows, groups = S.shape
    if groups != (int(K) + 31) // 32:
        raise GemmError(-3, f"scales have {groups} groups per row; K = {K} needs {(K + 31) // 32}")
    nbytes = mx_scales_b_size(rows, K) if for_b else mx_scales_size(rows, K)
    if out is None:
        out = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=S.device)
    elif out.numel() * out.element_size() < nbytes or out.device != S.device:
        raise GemmError(-3, "out is too small or on another device")
    ld = int(S.stride(0)) if rows > 1 else max(groups, 1)
    if rows > 0 and groups > 1 and S.stride(1) != 1:
        raise GemmError(-3, "scales: inner dimension must be contiguous")
    lib = load()
    fn = lib.gemm_mx_pack_scales_b if for_b else lib.gemm_mx_pack_scales
    st = fn(S.data_ptr(), rows, int(K), ld, out.data_ptr(), _stream_handle(stream, S.device))
    if st != 0:
        raise GemmError(st, "gemm_mx_pack_scales_b" if for_b else "gemm_mx_pack_scales")
    return out


def mx_pack_scales(S, K: int, out=None, *, stream=None):
    """The scales of A in the layout gemm_mx reads, from row-major ones: S is a
    CUDA uint8 tensor (M, ceil(K / 32)) of UE8M0 bytes (row stride free, inner
    stride 1).  Returns a uint8 tensor of mx_scales_size(M, K) bytes."""
    return _pack(S, K, out, stream, False)


def mx_pack_scales_b(S, K: int, out=None, *, stream=None):
    """The scales of B (N, ceil(K / 32)) in the layout gemm_mx reads (blocks
    for 224-column tiles); a uint8 tensor of mx_scales_b_size(N, K) bytes."""
    return _pack(S, K, out, stream, True)


def gemm_mx(A, B, SA, SB, D=None, *, fmt=None, out_dtype=None, alpha: float = 1.0,
            options=None, stream=None):
    """Block-scaled FP8: D[i, j] = alpha * sum_k (A[i, k] sa) (B[j, k] sb), one UE8M0
    scale per 32 K elements of each row.  A (M, K) and B (N, K) as for gemm_fp8;
    SA / SB the scales of A and B as mx_pack_scales / mx_pack_scales_b lay them
    out (uint8 CUDA tensors)."""
    import torch

    for t in (A, B, SA, SB):
        if t.device.type != "cuda":
            raise GemmError(-1, "operands must be CUDA tensors")
    code = _fp8_code(A, fmt)
    if _fp8_code(B, fmt) != code:
        raise GemmError(-2, "A and B must share an FP8 format")
    M, K = A.shape
    N, Kb = B.shape
    if Kb != K:
        raise GemmError(-3, f"K mismatch ({K} vs {Kb})")
    for t, need in ((SA, mx_scales_size(M, K)), (SB, mx_scales_b_size(N, K))):
        if t.dtype != torch.uint8 or t.numel() < need:
            raise GemmError(-3, "scales: uint8 tensors of mx_scales_size(M, K) and "
                                "mx_scales_b_size(N, K) bytes")
    odt = out_dtype if out_dtype is not None else (D.dtype if D is not None else torch.bfloat16)
    if D is None:
        D = torch.empty((M, N), dtype=odt, device=A.device)
    elif D.dtype != odt or tuple(D.shape) != (M, N):
        raise GemmError(-3, "D has the wrong dtype or shape")
    st = load().gemm_mx_run(A.data_ptr(), B.data_ptr(), SA.data_ptr(), SB.data_ptr(),
                            D.data_ptr(), M, N, K, _ld(A, 16), _ld(B, 16), _ld(D), code,
                            _dtype_code(D), float(alpha), _options(options),
                            _stream_handle(stream, A.device))
    if st != 0:
        raise GemmError(st, "gemm_mx_run")
    return D


def gemm_mx_plan(M: int, N: int, K: int, in_format: int = GEMM_E4M3, options=None) -> dict:
    """The tile shape and persistent grid gemm_mx would use on the current device."""
    vals = [ctypes.c_int() for _ in range(5)]
    tiles = ctypes.c_int64()
    group, order = ctypes.c_int(), ctypes.c_int()
    st = load().gemm_mx_plan(M, N, K, in_format, _options(options),
                             *[ctypes.byref(v) for v in vals], ctypes.byref(tiles),
                             ctypes.byref(group), ctypes.byref(order))
    if st != 0:
        raise GemmError(st, "gemm_mx_plan")
    keys = ("cta_group", "block_m", "block_n", "stages", "num_clusters")
    out = {k: v.value for k, v in zip(keys, vals)}
    out["num_tiles"] = tiles.value
    out["raster_group"] = group.value
    out["raster_order"] = order.value
    return out


def gemm_plan(M: int, N: int, K: int, dtype: int = GEMM_F16, layout: int = LAYOUT_ABT,
              options=None) -> dict:
    """The tile shape and persistent grid a call would use on the current device."""
    vals = [ctypes.c_int() for _ in range(5)]
    tiles = ctypes.c_int64()
    split, group, order, hints, ks = (ctypes.c_int() for _ in range(5))
    st = load().gemm_plan(M, N, K, dtype, layout, _options(options),
                          *[ctypes.byref(v) for v in vals], ctypes.byref(tiles),
                          ctypes.byref(split), ctypes.byref(group), ctypes.byref(order),
                          ctypes.byref(hints), ctypes.byref(ks))
    if st != 0:
        raise GemmError(st, "gemm_plan")
    keys = ("cta_group", "block_m", "block_n", "stages", "num_clusters")
    out = {k: v.value for k, v in zip(keys, vals)}
    out["num_tiles"] = tiles.value
    out["tail_split"] = split.value
    out["raster_group"] = group.value
    out["raster_order"] = order.value
    out["l2_hints"] = hints.value
    out["cluster_ksplit"] = ks.value
    return out


def gemm_tile_origin(M: int, N: int, block_m: int, block_n: int, group: int, task: int,
                     raster_order: int = 1):
    """(m0, n0) of the tile the persistent scheduler assigns to `task` (raster
    groups of `group` M tiles for raster_order 1, N tiles for 2)."""
    m0, n0 = ctypes.c_int64(), ctypes.c_int64()
    st = load().gemm_tile_origin(M, N, block_m, block_n, group, raster_order, task,
                                 ctypes.byref(m0), ctypes.byref(n0))
    if st != 0:
        raise GemmError(st, "gemm_tile_origin")
    return m0.value, n0.value


def gemm_device_status(clear: bool = True) -> int:
    """Synchronise and return the device error word (0 = no kernel wait gave up)."""
    v = ctypes.c_uint32()
    st = load().gemm_device_status(ctypes.byref(v), int(bool(clear)))
    if st != 0:
        raise GemmError(st, "gemm_device_status")
    return v.value


def gemm_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Launch the failure-path self-test (a bounded wait that must run out)."""
    import torch

    st = load().gemm_selftest_wait_timeout(int(limit_ns), _stream_handle(stream, torch.device("cuda")))
    if st != 0:
        raise GemmError(st, "gemm_selftest_wait_timeout")


def gemm_selftest_gemm_timeout(A, B, D, wait_limit_ns: int, *, layout: int = LAYOUT_ABT,
                               options=None, stream=None) -> None:
    """The GEMM kernel with every barrier wait limited to `wait_limit_ns`: a
    limit below the operands' arrival time makes a wait give up, which
    exercises the kernel's abort path (D is left unspecified)."""
    M, K = A.shape
    N = B.shape[0] if layout == LAYOUT_ABT else B.shape[1]
    if tuple(D.shape) != (M, N) or D.dtype != A.dtype or B.dtype != A.dtype:
        raise GemmError(-3, "D has the wrong dtype or shape")
    st = load().gemm_selftest_gemm_timeout(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                                           _ld(A), _ld(B), _ld(D), _dtype_code(A), int(layout),
                                           _options(options), int(wait_limit_ns),
                                           _stream_handle(stream, A.device))
    if st != 0:
        raise GemmError(st, "gemm_selftest_gemm_timeout")


def gemm_run_clock_probe(A, B, D, probe, *, layout: int = LAYOUT_ABT, options=None,
                         stream=None):
    """gemm_run on (A, B, D) that also writes the first CTA's start and end
    (%clock64, %globaltimer) into `probe`, an int64 CUDA tensor of 4 words."""
    M, K = A.shape
    N = B.shape[0] if layout == LAYOUT_ABT else B.shape[1]
    if tuple(D.shape) != (M, N) or D.dtype != A.dtype or B.dtype != A.dtype:
        raise GemmError(-3, "D has the wrong dtype or shape")
    if probe.device.type != "cuda" or probe.numel() < 4 or probe.element_size() != 8:
        raise GemmError(-1, "probe must be a CUDA tensor of at least four 8-byte words")
    st = load().gemm_run_clock_probe(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, _ld(A),
                                     _ld(B), _ld(D), _dtype_code(A), int(layout),
                                     _options(options), probe.data_ptr(),
                                     _stream_handle(stream, A.device))
    if st != 0:
        raise GemmError(st, "gemm_run_clock_probe")
    return D


def gemm_run_no_alloc(A, B, D, *, layout: int = LAYOUT_ABT, options=None, stream=None):
    """The GEMM through gemm_run_no_alloc: no allocation anywhere on the path.

    For callers that cannot allocate device memory at call time.  D must be
    given (the caller owns every buffer); the split tail uses the library's
    fixed scratch array.  Calls on different streams must not overlap.
    """
    if A.device.type != "cuda" or B.device.type != "cuda" or D.device.type != "cuda":
        raise GemmError(-1, "operands must be CUDA tensors")
    M, K = A.shape
    N = B.shape[0] if layout == LAYOUT_ABT else B.shape[1]
    if tuple(D.shape) != (M, N) or D.dtype != A.dtype or B.dtype != A.dtype:
        raise GemmError(-3, "D has the wrong dtype or shape")
    st = load().gemm_run_no_alloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, _ld(A),
                                  _ld(B), _ld(D), _dtype_code(A), int(layout), _options(options),
                                  _stream_handle(stream, A.device))
    if st != 0:
        raise GemmError(st, "gemm_run_no_alloc")
    return D


# The C entry points' names for the FP8 and block-scaled calls (the functions
# above take torch tensors; these are the same functions under the C names).
def gemm_fp8_run(A, B, D=None, *, fmt=None, out_dtype=None, alpha: float = 1.0, options=None,
                 stream=None, workspace="auto"):
    """gemm_fp8_run / gemm_fp8_run_workspace of the C ABI (see gemm_fp8)."""
    return gemm_fp8(A, B, D, fmt=fmt, out_dtype=out_dtype, alpha=alpha, options=options,
                    stream=stream, workspace=workspace)


def gemm_fp8_abt(A, B, D=None, *, fmt=None, out_dtype=None, alpha: float = 1.0, stream=None):
    """gemm_fp8_abt of the C ABI: gemm_fp8 with the default plan."""
    return gemm_fp8(A, B, D, fmt=fmt, out_dtype=out_dtype, alpha=alpha, stream=stream)


def gemm_mx_run(A, B, SA, SB, D=None, *, fmt=None, out_dtype=None, alpha: float = 1.0,
                options=None, stream=None):
    """gemm_mx_run of the C ABI (see gemm_mx)."""
    return gemm_mx(A, B, SA, SB, D, fmt=fmt, out_dtype=out_dtype, alpha=alpha, options=options,
                   stream=stream)


def gemm_mx_abt(A, B, SA, SB, D=None, *, fmt=None, out_dtype=None, alpha: float = 1.0,
                stream=None):
    """gemm_mx_abt of the C ABI: gemm_mx with the default plan."""
    return gemm_mx(A, B, SA, SB, D, fmt=fmt, out_dtype=out_dtype, alpha=alpha, stream=stream)


def gemm_run_workspace(A, B, D=None, *, layout: int = LAYOUT_ABT, options=None, stream=None,
                       workspace="auto"):
    """gemm_run_workspace of the C ABI: gemm_run, whose `workspace` argument is
    the caller's buffer (or "auto")."""
    return gemm_run(A, B, D, layout=layout, options=options, stream=stream, workspace=workspace)


gemm_fp8_run_workspace = gemm_fp8_run
gemm_mx_scales_size = mx_scales_size
gemm_mx_scales_b_size = mx_scales_b_size
gemm_mx_pack_scales = mx_pack_scales
gemm_mx_pack_scales_b = mx_pack_scales_b
