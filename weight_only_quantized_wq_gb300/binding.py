"""ctypes binding of libwq (include/wq.h): argument marshalling only.

Every function here forwards to the C entry point of the same name.  torch is
used for device memory and the current CUDA stream, nothing else; all the
arithmetic runs in the library's CUDA kernels.  If libwq.so is missing the
import fails -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libwq.so")

WQ_F16, WQ_BF16, WQ_F32 = 0, 1, 2
_DTYPE = {torch.float16: WQ_F16, torch.bfloat16: WQ_BF16, torch.float32: WQ_F32}

STATUS = ["WQ_OK", "WQ_ERR_NULL", "WQ_ERR_SHAPE", "WQ_ERR_WBIT", "WQ_ERR_GROUP", "WQ_ERR_DTYPE",
          "WQ_ERR_ALIGN", "WQ_ERR_WORKSPACE", "WQ_ERR_ARCH", "WQ_ERR_CUDA", "WQ_ERR_TIMEOUT"]

EXPORTS = ("wq_status_string", "wq_chunk_k", "wq_packed_bytes", "wq_pack", "wq_unpack",
           "wq_workspace_bytes", "wq_matmul", "wq_matmul_ex", "wq_matmul_noalloc", "wq_matmul_path",
           "wq_t2_pack", "wq_t2_workspace_bytes", "wq_t2_matmul", "wq_check_device")

PATHS = {0: "decode_kernel", 1: "midm_kernel", 2: "prefill_kernel", 3: "prefill_kernel"}

# the failure-path test hook of include/wq_testing.h
TESTING_EXPORTS = ("wq_testing_decode_timeout",)


class WQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = STATUS[status] if 0 <= status < len(STATUS) else str(status)
        super().__init__("%s: %s (%s)" % (what, name, wq_status_string(status)))


_lib = None


def lib() -> ctypes.CDLL:
    """Load libwq.so (built by weight_only_quantized_wq_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError("libwq.so is not built (run weight_only_quantized_wq_gb300.build.build())")
        L = ctypes.CDLL(_LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.wq_status_string.restype = ctypes.c_char_p
        L.wq_status_string.argtypes = [I]
        L.wq_chunk_k.restype = I
        L.wq_chunk_k.argtypes = [I]
        L.wq_packed_bytes.restype = Z
        L.wq_packed_bytes.argtypes = [I, I, I]
        L.wq_pack.restype = I
        L.wq_pack.argtypes = [P, I, I, I, P, P]
        L.wq_unpack.restype = I
        L.wq_unpack.argtypes = [P, I, I, I, P, P]
        L.wq_workspace_bytes.restype = Z
        L.wq_workspace_bytes.argtypes = [I, I, I, I, I]
        L.wq_matmul.restype = I
        L.wq_matmul.argtypes = [P, I, P, P, I, P, I, I, I, I, I, P, P, Z, P]
        L.wq_matmul_ex.restype = I
        L.wq_matmul_ex.argtypes = [P, I, P, P, I, P, I, I, I, I, I, P, I, P, Z, P]
        L.wq_matmul_noalloc.restype = I
        L.wq_matmul_noalloc.argtypes = [P, I, P, P, I, P, I, I, I, I, I, P, P]
        L.wq_t2_pack.restype = I
        L.wq_t2_pack.argtypes = [P, I, I, P, P]
        L.wq_t2_workspace_bytes.restype = Z
        L.wq_t2_workspace_bytes.argtypes = [I, I, I]
        L.wq_t2_matmul.restype = I
        L.wq_t2_matmul.argtypes = [P, P, I, I, I, P, P, Z, P]
        L.wq_matmul_path.restype = I
        L.wq_matmul_path.argtypes = [I, I, I, I, I, I, I]
        L.wq_testing_decode_timeout.restype = I
        L.wq_testing_decode_timeout.argtypes = [P, I, P, P, I, P, I, I, I, I, I, P, P, Z, ctypes.c_longlong, I, P]
        L.wq_check_device.restype = I
        L.wq_check_device.argtypes = [P]
        _lib = L
    return _lib


def _ptr(t):
    # plain ints: the c_void_p argtypes convert them (None is NULL)
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


def _check(st: int, what: str):
    if st != 0:
        raise WQError(st, what)


def wq_status_string(status: int) -> str:
    return lib().wq_status_string(int(status)).decode()


def wq_chunk_k(w_bit: int) -> int:
    return lib().wq_chunk_k(int(w_bit))


def wq_packed_bytes(K: int, N: int, w_bit: int) -> int:
    return lib().wq_packed_bytes(K, N, w_bit)


def wq_pack(q_in: torch.Tensor, K: int, N: int, w_bit: int, packed_out: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """Repack page-layout weights (int32 (K/pack, N), or int8 (N, K) for w_bit 8)
    into the tiled layout; returns the uint8 packed buffer."""
    if packed_out is None:
        n = wq_packed_bytes(K, N, w_bit)
        packed_out = torch.empty(max(n, 16), dtype=torch.uint8, device=q_in.device)
    _check(lib().wq_pack(_ptr(q_in), K, N, w_bit, _ptr(packed_out), _stream(stream)), "wq_pack")
    return packed_out


def wq_unpack(packed: torch.Tensor, K: int, N: int, w_bit: int, codes_out: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """Inverse of wq_pack: uint8 codes (K, N)."""
    if codes_out is None:
        codes_out = torch.empty((K, N), dtype=torch.uint8, device=packed.device)
    _check(lib().wq_unpack(_ptr(packed), K, N, w_bit, _ptr(codes_out), _stream(stream)), "wq_unpack")
    return codes_out


def wq_workspace_bytes(M: int, N: int, K: int, w_bit: int, group_size: int) -> int:
    return lib().wq_workspace_bytes(M, N, K, w_bit, group_size)


_workspaces: dict = {}
_needs: dict = {}


def workspace_for(M, N, K, w_bit, group_size, device) -> torch.Tensor | None:
    """A zero-filled workspace big enough for this problem, cached per device.
    Completed calls leave it reusable (its counters back at zero)."""
    dkey = torch.device(device).index
    nkey = (dkey, M, N, K, w_bit, group_size)
    need = _needs.get(nkey)
    if need is None:
        need = _needs[nkey] = wq_workspace_bytes(M, N, K, w_bit, group_size)
    if need == 0:
        return None
    ws = _workspaces.get(dkey)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(need, dtype=torch.uint8, device=device)
        _workspaces[dkey] = ws
    return ws


def wq_matmul(x: torch.Tensor, packed_w: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor | None,
              M: int, N: int, K: int, w_bit: int, group_size: int, out: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y (M, N) fp32 = x @ dequant(W) through the C entry point wq_matmul."""
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = workspace_for(M, N, K, w_bit, group_size, x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().wq_matmul(_ptr(x), _DTYPE.get(x.dtype, -1), _ptr(packed_w), _ptr(scales),
                         _DTYPE.get(scales.dtype, -1), _ptr(zeros), M, N, K, w_bit, group_size,
                         _ptr(out), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "wq_matmul")
    return out


def wq_matmul_ex(x: torch.Tensor, packed_w: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor | None,
                 M: int, N: int, K: int, w_bit: int, group_size: int, out: torch.Tensor | None = None,
                 out_dtype=torch.float32, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y (M, N) in out_dtype (fp32, fp16 or bf16) = x @ dequant(W), accumulated in fp32 and
    rounded once on store, through the C entry point wq_matmul_ex."""
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    if workspace is None:
        workspace = workspace_for(M, N, K, w_bit, group_size, x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().wq_matmul_ex(_ptr(x), _DTYPE.get(x.dtype, -1), _ptr(packed_w), _ptr(scales),
                            _DTYPE.get(scales.dtype, -1), _ptr(zeros), M, N, K, w_bit, group_size,
                            _ptr(out), _DTYPE.get(out.dtype, -1), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "wq_matmul_ex")
    return out


def wq_matmul_noalloc(x: torch.Tensor, packed_w: torch.Tensor, scales: torch.Tensor,
                      zeros: torch.Tensor | None, M: int, N: int, K: int, w_bit: int, group_size: int,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Same as wq_matmul, through the C entry point that uses the library's own
    fixed scratch instead of a caller workspace (no allocation on any call)."""
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    st = lib().wq_matmul_noalloc(_ptr(x), _DTYPE.get(x.dtype, -1), _ptr(packed_w), _ptr(scales),
                                 _DTYPE.get(scales.dtype, -1), _ptr(zeros), M, N, K, w_bit, group_size,
                                 _ptr(out), _stream(stream))
    _check(st, "wq_matmul_noalloc")
    return out


def wq_t2_pack(q_in: torch.Tensor, K: int, N: int, packed_out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """Repack Liger planar ternary bytes (K/4, N) uint8 into the tiled 2-bit layout."""
    if packed_out is None:
        packed_out = torch.empty(max(K * N // 4, 16), dtype=torch.uint8, device=q_in.device)
    _check(lib().wq_t2_pack(_ptr(q_in), K, N, _ptr(packed_out), _stream(stream)), "wq_t2_pack")
    return packed_out


def wq_t2_workspace_bytes(M: int, N: int, K: int) -> int:
    return lib().wq_t2_workspace_bytes(M, N, K)


_t2_workspaces: dict = {}


def wq_t2_matmul(x: torch.Tensor, packed_w: torch.Tensor, M: int, N: int, K: int,
                 out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """y (M, N) int32 = x (M, K) int8 @ ternary weights, through wq_t2_matmul."""
    if out is None:
        out = torch.empty((M, N), dtype=torch.int32, device=x.device)
    if workspace is None:
        need = wq_t2_workspace_bytes(M, N, K)
        dkey = torch.device(x.device).index
        workspace = _t2_workspaces.get(dkey)
        if need and (workspace is None or workspace.numel() < need):
            workspace = _t2_workspaces[dkey] = torch.zeros(need, dtype=torch.uint8, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel()
    st = lib().wq_t2_matmul(_ptr(x), _ptr(packed_w), M, N, K, _ptr(out), _ptr(workspace), ws_bytes,
                            _stream(stream))
    _check(st, "wq_t2_matmul")
    return out


def wq_matmul_path(M: int, N: int, K: int, w_bit: int, group_size: int, x_dtype, s_dtype) -> int:
    """Kernel family wq_matmul runs (0 few-token, 1 exact tensor-core, 2 many-token, 3 many-token
    with two-term weights; -1 invalid).  Dtypes are torch dtypes or the WQ_* codes."""
    xd = _DTYPE.get(x_dtype, x_dtype)
    sd = _DTYPE.get(s_dtype, s_dtype)
    return lib().wq_matmul_path(M, N, K, w_bit, group_size, int(xd), int(sd))


def wq_testing_decode_timeout(x: torch.Tensor, packed_w: torch.Tensor, scales: torch.Tensor,
                              zeros: torch.Tensor | None, M: int, N: int, K: int, w_bit: int, group_size: int,
                              wait_limit_cycles: int, withhold_stage: int, out: torch.Tensor | None = None,
                              workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The few-token kernel with a short barrier-wait limit and one withheld ring
    stage (include/wq_testing.h): the failure path, without any fault."""
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = workspace_for(M, N, K, w_bit, group_size, x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().wq_testing_decode_timeout(_ptr(x), _DTYPE.get(x.dtype, -1), _ptr(packed_w), _ptr(scales),
                                         _DTYPE.get(scales.dtype, -1), _ptr(zeros), M, N, K, w_bit, group_size,
                                         _ptr(out), _ptr(workspace), ws_bytes, int(wait_limit_cycles),
                                         int(withhold_stage), _stream(stream))
    _check(st, "wq_testing_decode_timeout")
    return out


def wq_check_device(stream=None) -> None:
    _check(lib().wq_check_device(_stream(stream)), "wq_check_device")
