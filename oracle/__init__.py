"""Plain fp64 CPU oracle of the Spark-X2.5 attention core.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never calls it and it never calls the CUDA library:
the two share no code.

The arithmetic lives in ``spark_oracle.c`` (plain C, fp64, OpenMP over rows).
This module only compiles it (with gcc, on first use or from ``build()``) and
marshals numpy arrays through ctypes.  Every function takes bf16 data as raw
16-bit patterns (``numpy.uint16``) so that the widening to fp64 is exact and
done in one place, the C file.

Sources (page title and section; see the C file for the formulas):
  * Spark-X2.5 architecture (4B / 1.7B): §1 config table, §2 hybrid attention
    masks, §3 head-wise output gate (Eq. 1), §4 layered RoPE table.
  * Spark-X2.5-4B hybrid-attention explainer (lshu.cn): the sliding layer's
    KV cache keeps only the latest 512 tokens.
  * Translated LLM-architecture notes, MiniMax-M2 chapter §13.3: partial RoPE.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spark_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libspark_oracle.so")

HEAD_DIM = 256
FULL = 0
SLIDING = 1

_lock = threading.Lock()
_default = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle C source into a shared object; return its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           "-std=c11", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(status: int, what: str):
    if status != 0:
        raise ValueError(f"{what}: oracle rejected its arguments (status {status})")


class OracleLib:
    """numpy front end of one compiled copy of the oracle C source."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_rope.argtypes = [P, P, i64, i32, f64, P]
        lib.oracle_rope.restype = i32
        lib.oracle_prefill.argtypes = [P, P, P, i32, i32, f64, i32, i32, i32, i32,
                                       i32, i32, P, i64, P]
        lib.oracle_prefill.restype = i32
        lib.oracle_decode.argtypes = [P, P, P, P, P, i64, i32, i32, f64, i32, i32,
                                      i32, i32, i32, P, P, P]
        lib.oracle_decode.restype = i32
        self.path = path
        self._lib = lib

    def rope(self, x: np.ndarray, pos: np.ndarray, rot_dim: int,
             theta: float) -> np.ndarray:
        """RoPE of head vectors x [n, 256] (fp64) at positions pos [n]."""
        x = _c(x, np.float64).reshape(-1, HEAD_DIM)
        pos = _c(pos, np.int32).reshape(-1)
        assert pos.shape[0] == x.shape[0]
        y = np.empty_like(x)
        _check(self._lib.oracle_rope(_ptr(x), _ptr(pos), x.shape[0], rot_dim,
                                     float(theta), _ptr(y)), "rope")
        return y

    def prefill(self, qkv_bits: np.ndarray, gate: np.ndarray, pos: np.ndarray,
                kind: int, window: int, theta: float, rot_dim: int, H: int, Hkv: int,
                rows: np.ndarray | None = None, gate_mode: int = 0) -> np.ndarray:
        """Oracle prefill.

        qkv_bits: uint16 [B, T, (H+2Hkv)*256] (bf16 patterns); gate: fp32
        [B, T, H]; pos: int32 [B, T].  rows: optional flat row ids (b*T + t).
        Returns fp64 [B, T, H*256] (all rows) or [len(rows), H*256].
        """
        qkv_bits = _c(qkv_bits, np.uint16)
        B, T, W = qkv_bits.shape
        assert W == (H + 2 * Hkv) * HEAD_DIM
        gate = _c(gate, np.float32).reshape(B, T, H)
        pos = _c(pos, np.int32).reshape(B, T)
        if rows is not None:
            rows = _c(rows, np.int64).reshape(-1)
            out = np.empty((rows.shape[0], H * HEAD_DIM), np.float64)
            n = rows.shape[0]
        else:
            out = np.empty((B, T, H * HEAD_DIM), np.float64)
            n = B * T
        _check(self._lib.oracle_prefill(_ptr(qkv_bits), _ptr(gate), _ptr(pos), kind,
                                        window, float(theta), rot_dim, gate_mode, B, T, H,
                                        Hkv, _ptr(rows), n, _ptr(out)), "prefill")
        return out

    def decode(self, qkv_bits: np.ndarray, gate: np.ndarray, pos: np.ndarray,
               k_cache_bits: np.ndarray, v_cache_bits: np.ndarray, kind: int,
               window: int, theta: float, rot_dim: int, H: int, Hkv: int,
               gate_mode: int = 0):
        """Oracle decode step (write-then-attend).

        qkv_bits: uint16 [B, (H+2Hkv)*256]; gate: fp32 [B, H]; pos: int32 [B];
        caches: uint16 [B, Hkv, cap, 256] holding post-RoPE keys / values
        BEFORE the step.  Returns (out fp64 [B, H*256], k_new fp64
        [B, Hkv, 256], v_new fp64 [B, Hkv, 256]); k_new / v_new are what the
        step stores at the slot of position pos.
        """
        qkv_bits = _c(qkv_bits, np.uint16)
        B = qkv_bits.shape[0]
        qkv_bits = qkv_bits.reshape(B, -1)
        assert qkv_bits.shape[1] == (H + 2 * Hkv) * HEAD_DIM
        gate = _c(gate, np.float32).reshape(B, H)
        pos = _c(pos, np.int32).reshape(B)
        k_cache_bits = _c(k_cache_bits, np.uint16)
        v_cache_bits = _c(v_cache_bits, np.uint16)
        assert k_cache_bits.shape == v_cache_bits.shape
        assert k_cache_bits.shape[0] == B and k_cache_bits.shape[1] == Hkv
        cap = k_cache_bits.shape[2]
        out = np.empty((B, H * HEAD_DIM), np.float64)
        k_new = np.empty((B, Hkv, HEAD_DIM), np.float64)
        v_new = np.empty((B, Hkv, HEAD_DIM), np.float64)
        _check(self._lib.oracle_decode(_ptr(qkv_bits), _ptr(gate), _ptr(pos),
                                       _ptr(k_cache_bits), _ptr(v_cache_bits), cap,
                                       kind, window, float(theta), rot_dim, gate_mode, B, H,
                                       Hkv, _ptr(out), _ptr(k_new), _ptr(v_new)), "decode")
        return out, k_new, v_new


def default() -> OracleLib:
    """The oracle built from spark_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
    return _default


def rope(*args, **kw):
    return default().rope(*args, **kw)


def prefill(*args, **kw):
    return default().prefill(*args, **kw)


def decode(*args, **kw):
    return default().decode(*args, **kw)


# ---------------------------------------------------------------- whole layer
#
# Spark-X2.5 architecture (4B / 1.7B), §3 Eq. 1 and Fig. 1: the attention
# block takes the normed hidden state x; q_k_v_proj (hidden -> (H+2Hkv)*256)
# and g_proj (hidden -> H, one gate logit per head) feed the core, and
# out_proj (H*256 -> hidden) maps the gated attention output back.  §1: the
# released checkpoints run in bfloat16, and §3: the gated output is cast back
# to the weight dtype.  Reading taken: every Linear's output is a bf16 tensor
# (rounded to nearest even from the exact product); the block output y is
# returned unrounded, in fp64.  No biases (the pages list none).


def bf16_round_bits(v: np.ndarray) -> np.ndarray:
    """fp64 values -> bf16 bit patterns, round to nearest even, exactly
    (no intermediate fp32 rounding).  Finite, normal-range inputs only."""
    v = np.asarray(v, np.float64)
    m, e = np.frexp(v)                      # v = m * 2^e, 0.5 <= |m| < 1
    q = np.rint(m * 256.0) / 256.0          # 8 significant bits, ties to even
    r = np.ldexp(q, e).astype(np.float32)   # exact in fp32
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp64 (exact)."""
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def layer_prefill(x_bits, w_qkv_bits, w_g_bits, w_o_bits, pos, kind, window, theta,
                  rot_dim, H, Hkv, rows=None, gate_mode=0):
    """Oracle of the attention block over a prefill.

    x_bits: uint16 [B, T, hidden]; w_qkv_bits [(H+2Hkv)*256, hidden];
    w_g_bits [H, hidden]; w_o_bits [hidden, H*256] (bf16 patterns, PyTorch
    Linear layout: y = x W^T); pos int32 [B, T].  rows: optional flat row ids
    (b*T + t) of y to compute.  Returns fp64 y [B, T, hidden] or
    [len(rows), hidden].
    """
    x = bits_to_f64(x_bits)
    B, T, hidden = x.shape
    qkv_bits = bf16_round_bits(x @ bits_to_f64(w_qkv_bits).T)          # q_k_v_proj
    g = bits_to_f64(bf16_round_bits(x @ bits_to_f64(w_g_bits).T))      # g_proj
    a = prefill(qkv_bits, g.astype(np.float32), pos, kind, window, theta, rot_dim, H, Hkv,
                rows=rows, gate_mode=gate_mode)                        # Eq. 1
    a = bits_to_f64(bf16_round_bits(a))                                # cast to bf16
    return a @ bits_to_f64(w_o_bits).T                                 # out_proj


def layer_decode(x_bits, w_qkv_bits, w_g_bits, w_o_bits, pos, k_cache_bits, v_cache_bits,
                 kind, window, theta, rot_dim, H, Hkv, gate_mode=0):
    """Oracle of the attention block for one decode step.

    x_bits: uint16 [B, hidden]; weights as in layer_prefill; pos int32 [B];
    caches uint16 [B, Hkv, cap, 256] BEFORE the step.  Returns (y fp64
    [B, hidden], k_new, v_new) with k_new / v_new as in decode().
    """
    x = bits_to_f64(x_bits).reshape(np.asarray(x_bits).shape[0], -1)
    qkv_bits = bf16_round_bits(x @ bits_to_f64(w_qkv_bits).T)
    g = bits_to_f64(bf16_round_bits(x @ bits_to_f64(w_g_bits).T))
    a, k_new, v_new = decode(qkv_bits, g.astype(np.float32), pos, k_cache_bits, v_cache_bits,
                             kind, window, theta, rot_dim, H, Hkv, gate_mode=gate_mode)
    a = bits_to_f64(bf16_round_bits(a))
    return a @ bits_to_f64(w_o_bits).T, k_new, v_new
