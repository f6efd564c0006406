"""fp64 CPU oracle for weight-absorbed MLA decode (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product library under ``mla_latent_decode_gb300/`` never imports, links or
calls it; the two share no code.  The arithmetic lives in ``mla_oracle.c``
(plain C, double precision); this module only builds it with gcc and
marshals numpy arrays into it.

Pages followed (cited by title and section):
  * "Resident VRAM: weights and KV cache", section on the KV ledger: one
    latent row per token of c_kv (512) + RoPE key (64), no head dimension.
  * "Kimi K3 decode on 2x8 B200: DP16 vs DP2 x DCP8", section "MLA: bytes
    conserved, DP16 kernel slowed by wave quantisation": partial (O, LSE)
    per token shard and an LSE-weighted merge; section "the problem: how to
    split": token-interleaved shards (slot p on rank p % 8).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None

ROW_DIM, NOPE_DIM, ROPE_DIM, VALUE_DIM = 576, 512, 64, 512


def build(force: bool = False) -> str:
    """Compile mla_oracle.c into libmla_oracle.so (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p, i32, i64, dbl = (ctypes.c_void_p, ctypes.c_int,
                                ctypes.c_int64, ctypes.c_double)
            lib.oracle_mla_decode_rows.restype = i32
            lib.oracle_mla_decode_rows.argtypes = [
                p, p, p, i32, p, p, i64, p, p, i32, i32, i32, dbl,
                p, i64, p, p, p, p]
            lib.oracle_lse_combine.restype = None
            lib.oracle_lse_combine.argtypes = [p, p, i32, i64, p, p]
            lib.oracle_gather.restype = None
            lib.oracle_gather.argtypes = [p, i32, p, i64, p, i32, p]
            lib.oracle_bf16_to_f64.restype = dbl
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_e4m3_to_f64.restype = dbl
            lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
            lib.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
            lib.oracle_kv_quantize.restype = None
            lib.oracle_kv_quantize.argtypes = [p, i64, p, p]
            lib.oracle_num_threads.restype = i32
            lib.oracle_num_threads.argtypes = []
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def bf16_to_f64(bits: int) -> float:
    return float(_load().oracle_bf16_to_f64(int(bits) & 0xFFFF))


def e4m3_to_f64(byte: int) -> float:
    return float(_load().oracle_e4m3_to_f64(int(byte) & 0xFF))


def f32_to_e4m3(v: float) -> int:
    """Nearest E4M3 code of a binary32 value (ties to even, saturated)."""
    return int(_load().oracle_f32_to_e4m3(float(v)))


def kv_quantize(rows):
    """FP8 cache write of binary32 rows [n, 576]: (codes uint8 [n, 576],
    scales fp32 [n]) with scale = fl32(amax / 448), code = E4M3(fl32(x /
    scale)); see oracle_kv_quantize."""
    x = _c(rows, np.float32).reshape(-1, ROW_DIM)
    n = x.shape[0]
    codes = np.zeros((n, ROW_DIM), np.uint8)
    scales = np.zeros((n,), np.float32)
    _load().oracle_kv_quantize(_ptr(x), n, _ptr(codes), _ptr(scales))
    return codes, scales


def _bf16_bits_to_f64(bits):
    """bf16 bit patterns (uint16 array) -> float64, exactly (the upper half
    of a binary32)."""
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def head_projection(x_bits, w_bits):
    """Per-head projection y[m, h, :] = x[m, h, :] . w[h] in fp64 over bf16
    inputs ([K3-MEM]: the query absorption q_nope . w_kc, and the output
    projection o_latent . w_vc): x [M, H, K], w [H, K, N] -> y [M, H, N]."""
    x = _bf16_bits_to_f64(x_bits)
    w = _bf16_bits_to_f64(w_bits)
    return np.einsum("mhk,hkn->mhn", x, w)


def mla_decode_rows(q_nope_bits, q_rope_bits, kv, kv_is_fp8, kv_scale,
                    req_to_token, seq_lens, kv_limit, B, q_len, H, sm_scale,
                    rows=None, row_lo=None, row_hi=None):
    """Oracle O (fp64 [n, 512]) and LSE (fp64 [n]) for the listed rows.

    Host numpy inputs, raw storage bits:
      q_nope_bits uint16 [B, q_len, H, 512], q_rope_bits uint16 [B, q_len, H, 64]
      kv uint16 [num_slots, 576] (bf16 bits) or uint8 (E4M3 bytes)
      kv_scale float32 [num_slots] or None; req_to_token int32 [B, stride]
      seq_lens int32 [B]; kv_limit int32 [B, q_len] or None
    ``rows`` are flat row ids (b * q_len + i) * H + h (default: all rows).
    ``row_lo``/``row_hi`` give a per-row token range (partial mode).
    """
    lib = _load()
    qn = _c(q_nope_bits, np.uint16)
    qr = _c(q_rope_bits, np.uint16)
    kvc = _c(kv, np.uint8 if kv_is_fp8 else np.uint16)
    ks = _c(kv_scale, np.float32)
    r2t = _c(req_to_token, np.int32)
    sl = _c(seq_lens, np.int32)
    kl = _c(kv_limit, np.int32)
    assert qn.size == B * q_len * H * NOPE_DIM and qr.size == B * q_len * H * ROPE_DIM
    assert r2t.ndim == 2 and r2t.shape[0] == B
    if kv_is_fp8:
        assert ks is not None and ks.size * ROW_DIM == kvc.size
    if rows is None:
        rows = np.arange(B * q_len * H, dtype=np.int64)
    rows = _c(rows, np.int64)
    n = rows.size
    lo = _c(row_lo, np.int64)
    hi = _c(row_hi, np.int64)
    O = np.zeros((n, VALUE_DIM), np.float64)
    lse = np.zeros(n, np.float64)
    rc = lib.oracle_mla_decode_rows(
        _ptr(qn), _ptr(qr), _ptr(kvc), int(bool(kv_is_fp8)), _ptr(ks),
        _ptr(r2t), r2t.shape[1], _ptr(sl), _ptr(kl), B, q_len, H,
        float(sm_scale), _ptr(rows), n, _ptr(lo), _ptr(hi), _ptr(O), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_mla_decode_rows failed: {rc}")
    return O, lse


def lse_combine(O_parts, lse_parts):
    """fp64 LSE merge: O_parts [P, rows, 512], lse_parts [P, rows]."""
    lib = _load()
    Op = _c(O_parts, np.float64)
    Lp = _c(lse_parts, np.float64)
    P, rows = Lp.shape
    assert Op.shape == (P, rows, VALUE_DIM)
    out = np.zeros((rows, VALUE_DIM), np.float64)
    lse = np.zeros(rows, np.float64)
    lib.oracle_lse_combine(_ptr(Op), _ptr(Lp), P, rows, _ptr(out), _ptr(lse))
    return out, lse


def gather(kv, req_to_token, seq_lens):
    """Raw-byte page gather: dense [sum(seq_lens), 576] copy of the rows."""
    lib = _load()
    kvc = np.ascontiguousarray(kv)
    elem = kvc.dtype.itemsize
    assert elem in (1, 2)
    r2t = _c(req_to_token, np.int32)
    sl = _c(seq_lens, np.int32)
    total = int(sl.astype(np.int64).sum())
    out = np.zeros((total, ROW_DIM), kvc.dtype)
    lib.oracle_gather(_ptr(kvc), elem, _ptr(r2t), r2t.shape[1], _ptr(sl),
                      int(sl.size), _ptr(out))
    return out
