"""ctypes binding of libspark_attn.so (include/spark_attn.h).

Argument marshalling only: every step of the attention core runs in the CUDA
library.  PyTorch supplies device memory and the current stream.  There is no
fallback: if the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

HEAD_DIM = 256

SPARK_OK = 0
SPARK_ERR_NULL = 1
SPARK_ERR_SHAPE = 2
SPARK_ERR_UNSUPPORTED = 3
SPARK_ERR_ALIGN = 4
SPARK_ERR_CAPACITY = 5
SPARK_ERR_WORKSPACE = 6
SPARK_ERR_CUDA = 7
SPARK_ERR_DEVICE = 8

SPARK_LAYER_FULL = 0
SPARK_LAYER_SLIDING = 1
SPARK_GATE_SIGMOID = 0
SPARK_GATE_SILU = 1

SPARK_NOALLOC_SCRATCH_BYTES = 8 << 20

SPARK_DEVERR_POSITION = 0x1
SPARK_DEVERR_TIMEOUT = 0x2


class spark_layer_desc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("window", ctypes.c_int32),
                ("rope_theta", ctypes.c_double), ("rot_dim", ctypes.c_int32),
                ("gate_mode", ctypes.c_int32)]


def _load() -> ctypes.CDLL:
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(
            f"the CUDA library {path} is not built; run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    D = ctypes.POINTER(spark_layer_desc)
    lib.spark_attn_prefill_workspace_size.argtypes = [i32, i32, i32, i32, D]
    lib.spark_attn_prefill_workspace_size.restype = sz
    lib.spark_attn_prefill.argtypes = [P, P, P, D, i32, i32, i32, i32, P, P, sz, P]
    lib.spark_attn_prefill.restype = i32
    lib.spark_attn_prefill_cache.argtypes = [P, P, P, P, P, i64, D, i32, i32, i32, i32, P, P,
                                             sz, P]
    lib.spark_attn_prefill_cache.restype = i32
    lib.spark_attn_prefill_chunk.argtypes = [P, P, P, P, P, i64, P, D, i32, i32, i32, i32, P, P,
                                             sz, P]
    lib.spark_attn_prefill_chunk.restype = i32
    lib.spark_attn_decode_workspace_size.argtypes = [i32, i32, i32, i64, D]
    lib.spark_attn_decode_workspace_size.restype = sz
    lib.spark_attn_decode_launch_count.argtypes = [i32, i32, i32, i64, D]
    lib.spark_attn_decode_launch_count.restype = i32
    lib.spark_attn_decode.argtypes = [P, P, P, P, P, i64, D, i32, i32, i32, P, P, sz, P]
    lib.spark_attn_decode.restype = i32
    lib.spark_attn_decode_noalloc.argtypes = [P, P, P, P, P, i64, D, i32, i32, i32, P, P, P]
    lib.spark_attn_decode_noalloc.restype = i32
    lib.spark_attn_prefill_host_workspace_size.argtypes = [i32, i32, i32, i32, D]
    lib.spark_attn_prefill_host_workspace_size.restype = sz
    lib.spark_attn_prefill_host.argtypes = [P, P, P, D, i32, i32, i32, i32, P, P, sz, P]
    lib.spark_attn_prefill_host.restype = i32
    lib.spark_attn_layer_prefill_workspace_size.argtypes = [i32, i32, i32, i32, i32, D]
    lib.spark_attn_layer_prefill_workspace_size.restype = sz
    lib.spark_attn_layer_prefill.argtypes = [P, P, P, P, P, P, P, i64, D, i32, i32, i32, i32,
                                             i32, P, P, sz, P]
    lib.spark_attn_layer_prefill.restype = i32
    lib.spark_attn_layer_decode_workspace_size.argtypes = [i32, i32, i32, i32, i64, D]
    lib.spark_attn_layer_decode_workspace_size.restype = sz
    lib.spark_attn_layer_decode.argtypes = [P, P, P, P, P, P, P, i64, D, i32, i32, i32, i32, P,
                                            P, sz, P]
    lib.spark_attn_layer_decode.restype = i32
    lib.spark_attn_linear.argtypes = [P, P, P, i64, i32, i32, P, P]
    lib.spark_attn_linear.restype = i32
    lib.spark_attn_read_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), i32, P]
    lib.spark_attn_read_status.restype = i32
    lib.spark_status_str.argtypes = [i32]
    lib.spark_status_str.restype = ctypes.c_char_p
    lib.spark_attn_version.argtypes = []
    lib.spark_attn_version.restype = ctypes.c_char_p
    return lib


lib = _load()


class SparkError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({spark_status_str(status)})")


class SparkDeviceFault(RuntimeError):
    """The kernels of a call recorded a device fault (SPARK_DEVERR_* bits)."""

    def __init__(self, bits: int, where: str):
        self.bits = bits
        super().__init__(f"{where}: device status 0x{bits:x}")


_check_own_workspace = False


def check_device_status(enabled: bool = True) -> None:
    """When enabled, a call that allocates its own workspace (workspace=None)
    reads that workspace's status word afterwards and raises SparkDeviceFault
    if it is not zero.  The read synchronizes the stream, so this is off by
    default; a caller that passes its own workspace reads it itself with
    spark_attn_read_status."""
    global _check_own_workspace
    _check_own_workspace = bool(enabled)


def _check_owned(workspace: torch.Tensor, where: str, stream) -> None:
    if _check_own_workspace:
        bits = spark_attn_read_status(workspace, stream=stream)
        if bits:
            raise SparkDeviceFault(bits, where)


def spark_status_str(status: int) -> str:
    return lib.spark_status_str(status).decode()


def spark_attn_version() -> str:
    return lib.spark_attn_version().decode()


def layer_desc(kind: int, window: int, rope_theta: float, rot_dim: int,
               gate_mode: int = SPARK_GATE_SIGMOID) -> spark_layer_desc:
    return spark_layer_desc(kind, window, float(rope_theta), rot_dim, gate_mode)


def as_desc(layer) -> spark_layer_desc:
    """Accepts a spark_layer_desc or any object with kind/window/theta/rot_dim."""
    if isinstance(layer, spark_layer_desc):
        return layer
    return layer_desc(layer.kind, layer.window, layer.theta, layer.rot_dim,
                      getattr(layer, "gate_mode", SPARK_GATE_SIGMOID))


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA {dtype} tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def spark_attn_prefill_workspace_size(B: int, T: int, H: int, Hkv: int, layer) -> int:
    d = as_desc(layer)
    return lib.spark_attn_prefill_workspace_size(B, T, H, Hkv, ctypes.byref(d))


def spark_attn_decode_workspace_size(B: int, H: int, Hkv: int, cap: int, layer) -> int:
    d = as_desc(layer)
    return lib.spark_attn_decode_workspace_size(B, H, Hkv, cap, ctypes.byref(d))


def spark_attn_decode_launch_count(B: int, H: int, Hkv: int, cap: int, layer) -> int:
    """Kernels one spark_attn_decode call enqueues (1 or 2; 0 if invalid)."""
    d = as_desc(layer)
    return lib.spark_attn_decode_launch_count(B, H, Hkv, cap, ctypes.byref(d))


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zeroed workspace: the header's status word and decode split counters
    must start at 0 (every call leaves the counters at 0 again)."""
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device or "cuda")


def spark_attn_prefill(qkv: torch.Tensor, gate: torch.Tensor, pos: torch.Tensor, layer,
                       out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """Prefill: qkv bf16 [B,T,(H+2Hkv)*256], gate fp32 [B,T,H], pos int32 [B,T]
    -> out bf16 [B,T,H*256]."""
    _need(qkv, torch.bfloat16, "qkv")
    _need(gate, torch.float32, "gate")
    _need(pos, torch.int32, "pos")
    B, T, W = qkv.shape
    H = gate.shape[-1]
    Hkv = (W // HEAD_DIM - H) // 2
    if gate.shape != (B, T, H) or pos.shape != (B, T) or (H + 2 * Hkv) * HEAD_DIM != W:
        raise ValueError("inconsistent prefill shapes")
    d = as_desc(layer)
    if out is None:
        out = torch.empty((B, T, H * HEAD_DIM), dtype=torch.bfloat16, device=qkv.device)
    _need(out, torch.bfloat16, "out")
    need = lib.spark_attn_prefill_workspace_size(B, T, H, Hkv, ctypes.byref(d))
    owned = workspace is None
    if owned:
        workspace = new_workspace(need, qkv.device)
    st = lib.spark_attn_prefill(_ptr(qkv), _ptr(gate), _ptr(pos), ctypes.byref(d), B, T, H,
                                Hkv, _ptr(out), _ptr(workspace), workspace.numel(),
                                _stream(stream))
    if st != SPARK_OK:
        raise SparkError(st, "spark_attn_prefill")
    if owned:
        _check_owned(workspace, "spark_attn_prefill", stream)
    return out


def spark_attn_prefill_cache(qkv: torch.Tensor, gate: torch.Tensor, pos: torch.Tensor,
                             k_cache: torch.Tensor, v_cache: torch.Tensor, layer,
                             out: torch.Tensor | None = None,
                             workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Prefill that also stores rotated K and V in the decode cache
    (caches bf16 [B,Hkv,cap,256]; see spark_attn_prefill for the rest)."""
    _need(qkv, torch.bfloat16, "qkv")
    _need(gate, torch.float32, "gate")
    _need(pos, torch.int32, "pos")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    B, T, W = qkv.shape
    H = gate.shape[-1]
    Hkv = (W // HEAD_DIM - H) // 2
    if (gate.shape != (B, T, H) or pos.shape != (B, T) or (H + 2 * Hkv) * HEAD_DIM != W
            or k_cache.shape != v_cache.shape or k_cache.shape[:2] != (B, Hkv)
            or k_cache.shape[3] != HEAD_DIM):
        raise ValueError("inconsistent prefill shapes")
    d = as_desc(layer)
    if out is None:
        out = torch.empty((B, T, H * HEAD_DIM), dtype=torch.bfloat16, device=qkv.device)
    _need(out, torch.bfloat16, "out")
    need = lib.spark_attn_prefill_workspace_size(B, T, H, Hkv, ctypes.byref(d))
    owned = workspace is None
    if owned:
        workspace = new_workspace(need, qkv.device)
    st = lib.spark_attn_prefill_cache(_ptr(qkv), _ptr(gate), _ptr(pos), _ptr(k_cache),
                                      _ptr(v_cache), k_cache.shape[2], ctypes.byref(d), B, T, H,
                                      Hkv, _ptr(out), _ptr(workspace), workspace.numel(),
                                      _stream(stream))
    if st != SPARK_OK:
        raise SparkError(st, "spark_attn_prefill_cache")
    if owned:
        _check_owned(workspace, "spark_attn_prefill_cache", stream)
    return out


def spark_attn_prefill_chunk(qkv: torch.Tensor, gate: torch.Tensor, pos: torch.Tensor,
                             k_cache: torch.Tensor, v_cache: torch.Tensor, start: torch.Tensor,
                             layer, out: torch.Tensor | None = None,
                             workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Chunked prefill: T more tokens per sequence on top of start[b] cached
    tokens (start: CUDA int32 [B]); see the C header for the cache rules."""
    _need(qkv, torch.bfloat16, "qkv")
    _need(gate, torch.float32, "gate")
    _need(pos, torch.int32, "pos")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(start, torch.int32, "start")
    B, T, W = qkv.shape
    H = gate.shape[-1]
    Hkv = (W // HEAD_DIM - H) // 2
    if (gate.shape != (B, T, H) or pos.shape != (B, T) or (H + 2 * Hkv) * HEAD_DIM != W
            or start.shape != (B,) or k_cache.shape != v_cache.shape
            or k_cache.shape[:2] != (B, Hkv) or k_cache.shape[3] != HEAD_DIM):
        raise ValueError("inconsistent chunked-prefill shapes")
    d = as_desc(layer)
    if out is None:
        out = torch.empty((B, T, H * HEAD_DIM), dtype=torch.bfloat16, device=qkv.device)
    _need(out, torch.bfloat16, "out")
    need = lib.spark_attn_prefill_workspace_size(B, T, H, Hkv, ctypes.byref(d))
    owned = workspace is None
    if owned:
        workspace = new_workspace(need, qkv.device)
    st = lib.spark_attn_prefill_chunk(_ptr(qkv), _ptr(gate), _ptr(pos), _ptr(k_cache),
                                      _ptr(v_cache), k_cache.shape[2], _ptr(start),
                                      ctypes.byref(d), B, T, H, Hkv, _ptr(out), _ptr(workspace),
                                      workspace.numel(), _stream(stream))
    if st != SPARK_OK:
        raise SparkError(st, "spark_attn_prefill_chunk")
    if owned:
        _check_owned(workspace, "spark_attn_prefill_chunk", stream)
    return out


def spark_attn_decode(qkv: torch.Tensor, gate: torch.Tensor, pos: torch.Tensor,
                      k_cache: torch.Tensor, v_cache: torch.Tensor, layer,
                      out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """One decode step: qkv bf16 [B,(H+2Hkv)*256], gate fp32 [B,H], pos int32 [B],
    caches bf16 [B,Hkv,cap,256] (updated in place) -> out bf16 [B,H*256]."""
    _need(qkv, torch.bfloat16, "qkv")
    _need(gate, torch.float32, "gate")
    _need(pos, torch.int32, "pos")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    B, W = qkv.shape
    H = gate.shape[-1]
    Hkv = (W // HEAD_DIM - H) // 2
    if (gate.shape != (B, H) or pos.shape != (B,) or k_cache.shape != v_cache.shape
            or k_cache.shape[:2] != (B, Hkv) or k_cache.shape[3] != HEAD_DIM):
        raise ValueError("inconsistent decode shapes")
    cap = k_cache.shape[2]
    d = as_desc(layer)
    if out is None:
        out = torch.empty((B, H * HEAD_DIM), dtype=torch.bfloat16, device=qkv.device)
    _need(out, torch.bfloat16, "out")
    need = lib.spark_attn_decode_workspace_size(B, H, Hkv, cap, ctypes.byref(d))
    owned = workspace is None
    if owned:
        workspace = new_workspace(need, qkv.device)
    st = lib.spark_attn_decode(_ptr(qkv), _ptr(gate), _ptr(pos), _ptr(k_cache), _ptr(v_cache),
                               cap, ctypes.byref(d), B, H, Hkv, _ptr(out), _ptr(workspace),
                               workspace.numel(), _stream(stream))
    if st != SPARK_OK:
        raise SparkError(st, "spark_attn_decode")
    if owned:
        _check_owned(workspace, "spark_attn_decode", stream)
    return out


def spark_attn_decode_noalloc(qkv: torch.Tensor, gate: torch.Tensor, pos: torch.Tensor,
                              k_cache: torch.Tensor, v_cache: torch.Tensor, layer,
                              out: torch.Tensor | None = None,
                              device_status: torch.Tensor | None = None,
                              stream=None) -> torch.Tensor:
    """spark_attn_decode without a workspace, for callers that cannot allocate
    one: the split-KV scratch is a fixed buffer inside the library (see the
    C header).  device_status: optional CUDA int32/uint32 tensor of one element
    that receives the device fault bits."""
    _need(qkv, torch.bfloat16, "qkv")
    _need(gate, torch.float32, "gate")
    _need(pos, torch.int32, "pos")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    B, W = qkv.shape
    H = gate.shape[-1]
    Hkv = (W // HEAD_DIM - H) // 2
    if (gate.shape != (B, H) or pos.shape != (B,) or k_cache.shape != v_cache.shape
            or k_cache.shape[:2] != (B, Hkv) or k_cache.shape[3] != HEAD_DIM):
        raise ValueError("inconsistent decode shapes")
    if device_status is not None and (not device_status.is_cuda or device_status.numel() != 1
                                      or device_status.element_size() != 4):
        raise ValueError("device_status must be a one-element 32-bit CUDA tensor")
    d = as_desc(layer)
    if out is None:
        out = torch.empty((B, H * HEAD_DIM), dtype=torch.bfloat16, device=qkv.device)
    _need(out, torch.bfloat16, "out")
    st = lib.spark_attn_decode_noalloc(_ptr(qkv), _ptr(gate), _ptr(pos), _ptr(k_cache),
                                       _ptr(v_cache), k_cache.shape[2], ctypes.byref(d), B, H,
                                       Hkv, _ptr(out), _ptr(device_status), _stream(stream))
    if st != SPARK_OK:
        raise SparkError(st, "spark_attn_decode_noalloc")
    return out


def spark_attn_linear(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor | None = None,
                      device_status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y = x W^T on the library's tcgen05 GEMM: x bf16 [..., K], w bf16 [N, K]
    (Linear layout) -> y bf16 [..., N].  device_status: one-element 32-bit
    CUDA tensor receiving SPARK_DEVERR_TIMEOUT (a fresh zeroed one if None;
    with check_device_status on, that one is read and a fault raised)."""
    _need(x, torch.bfloat16, "x")
    _need(w, torch.bfloat16, "w")
    N, K = w.shape
    if x.shape[-1] != K:
        raise ValueError("x and w disagree on K")
    M = x.numel() // K if K else 0
    if y is None:
        y = torch.empty((*x.shape[:-1], N), dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, "y")
    if y.shape != (*x.shape[:-1], N):
        raise ValueError("y has the wrong shape")
    owned = device_status is None
    if owned:
        device_status = torch.zeros(1, dtype=torch.int32, device=x.device)
    if not device_status.is_cuda or device_status.numel() != 1 or device_status.element_size() != 4:
        raise ValueError("device_status must be a one-element 32-bit CUDA tensor")
    st = lib.spark_attn_linear(_ptr(x), _ptr(w), _ptr(y), M, N, K, _ptr(device_status),
                               _stream(stream))
    if st != SPARK_OK:
        raise SparkError(st, "spark_attn_linear")
    if owned and _check_own_workspace:
        bits = int(device_status.item())
        if bits:
            raise SparkDeviceFault(bits, "spark_attn_linear")
    return y


def _need_host(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or t.is_cuda:
        raise TypeError(f"{name} must be a host (CPU) {dtype} tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def spark_attn_prefill_host_workspace_size(B: int, T: int, H: int, Hkv: int, layer) -> int:
    d = as_desc(layer)
    return lib.spark_attn_prefill_host_workspace_size(B, T, H, Hkv, ctypes.byref(d))


def spark_attn_prefill_host(qkv: torch.Tensor, gate: torch.Tensor, pos: torch.Tensor, layer,
                            out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                            stream=None, device=None) -> torch.Tensor:
    """Prefill of HOST tensors (pin them for overlapped copies): qkv bf16
    [B,T,(H+2Hkv)*256], gate fp32 [B,T,H], pos int32 [B,T] -> out bf16
    [B,T,H*256] in host memory.  The copies of one sequence overlap the
    compute of another; synchronize `stream` before reading `out`."""
    _need_host(qkv, torch.bfloat16, "qkv")
    _need_host(gate, torch.float32, "gate")
    _need_host(pos, torch.int32, "pos")
    B, T, W = qkv.shape
    H = gate.shape[-1]
    Hkv = (W // HEAD_DIM - H) // 2
    if gate.shape != (B, T, H) or pos.shape != (B, T) or (H + 2 * Hkv) * HEAD_DIM != W:
        raise ValueError("inconsistent prefill shapes")
    d = as_desc(layer)
    if out is None:
        out = torch.empty((B, T, H * HEAD_DIM), dtype=torch.bfloat16, pin_memory=qkv.is_pinned())
    _need_host(out, torch.bfloat16, "out")
    need = lib.spark_attn_prefill_host_workspace_size(B, T, H, Hkv, ctypes.byref(d))
    owned = workspace is None
    if owned:
        workspace = new_workspace(need, device)
    st = lib.spark_attn_prefill_host(_ptr(qkv), _ptr(gate), _ptr(pos), ctypes.byref(d), B, T, H,
                                     Hkv, _ptr(out), _ptr(workspace), workspace.numel(),
                                     _stream(stream))
    if st != SPARK_OK:
        raise SparkError(st, "spark_attn_prefill_host")
    if owned:
        _check_owned(workspace, "spark_attn_prefill_host", stream)
    return out


def _layer_weights(w_qkv, w_g, w_o, hidden: int):
    for t, name in ((w_qkv, "w_qkv"), (w_g, "w_g"), (w_o, "w_o")):
        _need(t, torch.bfloat16, name)
    H = w_g.shape[0]
    Hkv = (w_qkv.shape[0] // HEAD_DIM - H) // 2
    if (w_g.shape != (H, hidden) or w_qkv.shape != ((H + 2 * Hkv) * HEAD_DIM, hidden)
            or w_o.shape != (hidden, H * HEAD_DIM)):
        raise ValueError("inconsistent projection weight shapes")
    return H, Hkv


def spark_attn_layer_prefill_workspace_size(B: int, T: int, hidden: int, H: int, Hkv: int,
                                            layer) -> int:
    d = as_desc(layer)
    return lib.spark_attn_layer_prefill_workspace_size(B, T, hidden, H, Hkv, ctypes.byref(d))


def spark_attn_layer_decode_workspace_size(B: int, hidden: int, H: int, Hkv: int, cap: int,
                                           layer) -> int:
    d = as_desc(layer)
    return lib.spark_attn_layer_decode_workspace_size(B, hidden, H, Hkv, cap, ctypes.byref(d))


def spark_attn_layer_prefill(x: torch.Tensor, w_qkv: torch.Tensor, w_g: torch.Tensor,
                             w_o: torch.Tensor, pos: torch.Tensor, layer,
                             k_cache: torch.Tensor | None = None,
                             v_cache: torch.Tensor | None = None,
                             y: torch.Tensor | None = None,
                             workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The attention block over a prefill: x bf16 [B,T,hidden] (normed hidden
    state), Linear weights w_qkv [(H+2Hkv)*256, hidden], w_g [H, hidden],
    w_o [hidden, H*256], pos int32 [B,T] -> y bf16 [B,T,hidden].  With caches
    (bf16 [B,Hkv,cap,256]) it also fills the decode cache."""
    _need(x, torch.bfloat16, "x")
    _need(pos, torch.int32, "pos")
    B, T, hidden = x.shape
    H, Hkv = _layer_weights(w_qkv, w_g, w_o, hidden)
    if pos.shape != (B, T):
        raise ValueError("inconsistent layer prefill shapes")
    cap = 0
    if k_cache is not None or v_cache is not None:
        _need(k_cache, torch.bfloat16, "k_cache")
        _need(v_cache, torch.bfloat16, "v_cache")
        if (k_cache.shape != v_cache.shape or k_cache.shape[:2] != (B, Hkv)
                or k_cache.shape[3] != HEAD_DIM):
            raise ValueError("inconsistent cache shapes")
        cap = k_cache.shape[2]
    d = as_desc(layer)
    if y is None:
        y = torch.empty((B, T, hidden), dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, "y")
    need = lib.spark_attn_layer_prefill_workspace_size(B, T, hidden, H, Hkv, ctypes.byref(d))
    owned = workspace is None
    if owned:
        workspace = new_workspace(need, x.device)
    st = lib.spark_attn_layer_prefill(_ptr(x), _ptr(w_qkv), _ptr(w_g), _ptr(w_o), _ptr(pos),
                                      _ptr(k_cache), _ptr(v_cache), cap, ctypes.byref(d), B, T,
                                      hidden, H, Hkv, _ptr(y), _ptr(workspace), workspace.numel(),
                                      _stream(stream))
    if st != SPARK_OK:
        raise SparkError(st, "spark_attn_layer_prefill")
    if owned:
        _check_owned(workspace, "spark_attn_layer_prefill", stream)
    return y


def spark_attn_layer_decode(x: torch.Tensor, w_qkv: torch.Tensor, w_g: torch.Tensor,
                            w_o: torch.Tensor, pos: torch.Tensor, k_cache: torch.Tensor,
                            v_cache: torch.Tensor, layer, y: torch.Tensor | None = None,
                            workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The attention block for one decode step: x bf16 [B,hidden], weights as
    for spark_attn_layer_prefill, pos int32 [B], caches bf16 [B,Hkv,cap,256]
    (updated in place) -> y bf16 [B,hidden]."""
    _need(x, torch.bfloat16, "x")
    _need(pos, torch.int32, "pos")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    B, hidden = x.shape
    H, Hkv = _layer_weights(w_qkv, w_g, w_o, hidden)
    if (pos.shape != (B,) or k_cache.shape != v_cache.shape or k_cache.shape[:2] != (B, Hkv)
            or k_cache.shape[3] != HEAD_DIM):
        raise ValueError("inconsistent layer decode shapes")
    cap = k_cache.shape[2]
    d = as_desc(layer)
    if y is None:
        y = torch.empty((B, hidden), dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, "y")
    need = lib.spark_attn_layer_decode_workspace_size(B, hidden, H, Hkv, cap, ctypes.byref(d))
    owned = workspace is None
    if owned:
        workspace = new_workspace(need, x.device)
    st = lib.spark_attn_layer_decode(_ptr(x), _ptr(w_qkv), _ptr(w_g), _ptr(w_o), _ptr(pos),
                                     _ptr(k_cache), _ptr(v_cache), cap, ctypes.byref(d), B, hidden,
                                     H, Hkv, _ptr(y), _ptr(workspace), workspace.numel(),
                                     _stream(stream))
    if st != SPARK_OK:
        raise SparkError(st, "spark_attn_layer_decode")
    if owned:
        _check_owned(workspace, "spark_attn_layer_decode", stream)
    return y


def spark_attn_read_status(workspace: torch.Tensor, clear: bool = False, stream=None) -> int:
    """The sticky device status word of a workspace (synchronizes)."""
    v = ctypes.c_uint32(0)
    st = lib.spark_attn_read_status(_ptr(workspace), ctypes.byref(v), int(clear),
                                    _stream(stream))
    if st != SPARK_OK:
        raise SparkError(st, "spark_attn_read_status")
    return v.value
