"""GB300 (sm_103a) MLA latent decode: thin Python binding of libmla_decode.so.

Every function here only marshals arguments (torch tensors -> device
pointers, the current CUDA stream) into the C ABI declared in
include/mla_decode.h; all arithmetic runs in the library's CUDA kernels.
There is no CPU fallback: if the library is missing, loading it raises.

    import mla_latent_decode_gb300 as mla
    O_part, LSE_part = mla.decode_partial(q_nope, q_rope, kv, ..., num_splits)
    out, lse = mla.lse_combine(O_part, LSE_part)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_decode.so")
ROW_DIM, NOPE_DIM, ROPE_DIM, VALUE_DIM, PAGE_SIZE = 576, 512, 64, 512, 64
KV_BF16, KV_FP8_E4M3 = 0, 1
_KV_DTYPE = {"bf16": KV_BF16, "fp8_e4m3": KV_FP8_E4M3}
ROWS_PER_UNIT = 256  # query rows per work unit of the BF16 tensor-core kernel
STATUS_WAIT_TIMEOUT, STATUS_BAD_LENGTH, STATUS_BAD_SLOT, STATUS_BAD_WORK = 1, 2, 4, 8

_lib = None
_lock = threading.Lock()


class MlaError(RuntimeError):
    """A non-zero return code of the C library, with its message."""

    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} (code {code})")
        self.code = code


def library() -> ctypes.CDLL:
    """Load libmla_decode.so (built by ``build.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        p, i32, i64, f32, f64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                 ctypes.c_float, ctypes.c_double)
        sig = {
            "mla_last_error_string": (ctypes.c_char_p, []),
            "mla_num_sms": (i32, [i32]),
            "mla_cluster_slots": (i32, []),
            "mla_plan_heuristic": (i32, [i32, i32]),
            "mla_plan_ex": (i32, [i32, i32, i32, i32, p, i32, i32, f64, f64, p, p, p]),
            "mla_plan": (i32, [i32, i32, i32, i32, i32, p, i32, p, p]),
            "mla_plan_parts_ex": (i32, [i32, i32, i32, i32, p, i32, i32, i32, f64,
                                        f64, p, p, p, p]),
            "mla_plan_parts": (i32, [i32, i32, i32, i32, i32, p, i32, i32, p, p,
                                     p]),
            "mla_plan_sched_ex": (i32, [i32, i32, i32, i32, p, i32, i32, i32, f64,
                                        f64, p, p, p, i64, p, p, p]),
            "mla_plan_sched": (i32, [i32, i32, i32, i32, i32, p, i32, i32, p, p,
                                     p, i64, p, p]),
            "mla_check_page_table": (i32, [p, i64, p, p, i32, i32, i32, i64]),
            "mla_decode_partial": (i32, [p, p, p, p, i32, i64, p, i64, p, p, i32,
                                         i32, i32, i32, i32, f32, i32, p, p, i32,
                                         p, p, p, p]),
            "mla_decode_partial_bf16_parts": (i32, [p, p, p, p, i32, i64, p, i64, p,
                                                    p, i32, i32, i32, i32, i32, f32,
                                                    i32, p, p, i32, p, p, p, p]),
            "mla_decode_partial_simt": (i32, [p, p, p, p, i32, i64, p, i64, p, p,
                                              i32, i32, i32, i32, i32, f32, i32, p,
                                              p, p, p, p]),
            "mla_decode": (i32, [p, p, p, p, i32, i64, p, i64, p, p, i32, i32,
                                 i32, i32, i32, f32, i32, p, p, i32, p, p, p, p,
                                 p, p, p]),
            "mla_decode_scratch": (i32, [p, p, p, p, i32, i64, p, i64, p, p, i32,
                                         i32, i32, i32, i32, f32, i32, p, p, i32,
                                         p, p, p, p]),
            "mla_scratch_bytes": (i64, [i32, i32, i32, i32, i32]),
            "mla_kv_write": (i32, [p, i64, p, p, i32, p, i64, p, p]),
            "mla_absorb_q": (i32, [p, p, p, i32, i32, p, p]),
            "mla_project_out": (i32, [p, p, p, i32, i32, p, p]),
            "mla_lse_combine": (i32, [p, p, i32, i64, p, p, p]),
            "mla_lse_combine_bf16_parts": (i32, [p, p, i32, i64, p, p, p]),
            "mla_debug_gather": (i32, [p, i32, i64, p, i64, p, p, i32, i32, p, p]),
            "mla_debug_wait": (i32, [i32, i32, p, p, p]),
            "mla_debug_quotients": (i32, [p, p, p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(rc: int) -> int:
    if rc < 0:
        raise MlaError(rc, library().mla_last_error_string().decode())
    return rc


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _on(t: torch.Tensor):
    """Make the tensor's device current for a call: the library launches
    on (and looks up per-device state for) the current device."""
    return torch.cuda.device(t.device)


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _host_i32(x) -> "ctypes.Array":
    vals = [int(v) for v in (x.tolist() if torch.is_tensor(x) else x)]
    return (ctypes.c_int32 * len(vals))(*vals)


# ------------------------------------------------------------------ planning
def num_sms(device: int = 0) -> int:
    return _check(library().mla_num_sms(device))


def cluster_slots() -> int:
    """Concurrently resident work units (4-CTA clusters) of the tensor-core
    decode kernel on this device."""
    return _check(library().mla_cluster_slots())


def plan_heuristic(B: int, q_len: int) -> int:
    """The pages' split rule max(1, min(148 // B // (2 q_len), 32))."""
    return _check(library().mla_plan_heuristic(B, q_len))


def plan_ex(seq_lens: Sequence[int], q_len: int, H: int, slots: int,
            s_max: int = 64, c0: float = 32.0, lam: float = 1.0,
            rows_per_unit: int = ROWS_PER_UNIT):
    """Wave-rounding planner: returns (num_splits, wave_eff, makespan)."""
    arr = _host_i32(seq_lens)
    S, eff, ms = ctypes.c_int(), ctypes.c_float(), ctypes.c_double()
    _check(library().mla_plan_ex(len(arr), q_len, H, rows_per_unit, arr,
                                 slots, s_max, float(c0), float(lam),
                                 ctypes.byref(S), ctypes.byref(eff),
                                 ctypes.byref(ms)))
    return S.value, eff.value, ms.value


def plan(B: int, q_len: int, H: int, seq_lens, num_shards: int = 1,
         num_sms: int = 0, kv_dtype: str = "bf16"):
    """Planner with the library defaults for the kernel that serves
    `kv_dtype`; num_sms=0 asks the device."""
    arr = _host_i32(seq_lens)
    assert len(arr) == B * num_shards
    S, eff = ctypes.c_int(), ctypes.c_float()
    _check(library().mla_plan(B, q_len, H, num_shards, _KV_DTYPE[kv_dtype],
                              arr, num_sms, ctypes.byref(S), ctypes.byref(eff)))
    return S.value, eff.value


def plan_parts_ex(seq_lens: Sequence[int], q_len: int, H: int, slots: int,
                  s_max: int = 64, max_parts: int = 8, c0: float = 32.0,
                  lam: float = 1.0, rows_per_unit: int = ROWS_PER_UNIT):
    """Per-request split planner: returns (S, boundaries np.int32 [V, S+1],
    wave_eff, makespan)."""
    import numpy as np
    arr = _host_i32(seq_lens)
    V = len(arr)
    out = (ctypes.c_int32 * (V * (s_max + 1)))()
    S, eff, ms = ctypes.c_int(), ctypes.c_float(), ctypes.c_double()
    _check(library().mla_plan_parts_ex(V, q_len, H, rows_per_unit, arr, slots,
                                       s_max, max_parts, float(c0), float(lam),
                                       out, ctypes.byref(S), ctypes.byref(eff),
                                       ctypes.byref(ms)))
    bnd = np.frombuffer(out, dtype=np.int32)[:V * (S.value + 1)]
    return S.value, bnd.reshape(V, S.value + 1).copy(), eff.value, ms.value


def plan_parts(B: int, q_len: int, H: int, seq_lens, num_shards: int = 1,
               num_sms: int = 0, kv_dtype: str = "bf16", max_parts: int = 8):
    """Per-request split planner with the library defaults for the kernel
    that serves `kv_dtype`: returns (S, boundaries np.int32 [V, S+1],
    wave_eff); num_sms=0 asks the device."""
    import numpy as np
    arr = _host_i32(seq_lens)
    V = len(arr)
    assert V == B * num_shards
    out = (ctypes.c_int32 * (V * 65))()
    S, eff = ctypes.c_int(), ctypes.c_float()
    _check(library().mla_plan_parts(B, q_len, H, num_shards, _KV_DTYPE[kv_dtype],
                                    arr, num_sms, max_parts, out,
                                    ctypes.byref(S), ctypes.byref(eff)))
    bnd = np.frombuffer(out, dtype=np.int32)[:V * (S.value + 1)]
    return S.value, bnd.reshape(V, S.value + 1).copy(), eff.value


def plan_sched_ex(seq_lens: Sequence[int], q_len: int, H: int, slots: int,
                  s_max: int = 64, max_parts: int = 8, c0: float = 32.0,
                  lam: float = 1.0, rows_per_unit: int = ROWS_PER_UNIT):
    """Work-balanced scheduler: returns (S, boundaries np.int32 [V, S+1],
    work np.int32 [V*S*U] (unit ids, longest first), wave_eff, makespan)."""
    import numpy as np
    arr = _host_i32(seq_lens)
    V = len(arr)
    U = -(-q_len * H // rows_per_unit)
    cap = V * s_max * U
    bnd_out = (ctypes.c_int32 * (V * (s_max + 1)))()
    work_out = (ctypes.c_int32 * cap)()
    S, n = ctypes.c_int(), ctypes.c_int64()
    eff, ms = ctypes.c_float(), ctypes.c_double()
    _check(library().mla_plan_sched_ex(V, q_len, H, rows_per_unit, arr, slots,
                                       s_max, max_parts, float(c0), float(lam),
                                       bnd_out, ctypes.byref(S), work_out, cap,
                                       ctypes.byref(n), ctypes.byref(eff),
                                       ctypes.byref(ms)))
    bnd = np.frombuffer(bnd_out, dtype=np.int32)[:V * (S.value + 1)]
    work = np.frombuffer(work_out, dtype=np.int32)[:n.value].copy()
    return S.value, bnd.reshape(V, S.value + 1).copy(), work, eff.value, ms.value


def plan_sched(B: int, q_len: int, H: int, seq_lens, num_shards: int = 1,
               num_sms: int = 0, kv_dtype: str = "bf16", max_parts: int = 8):
    """Work-balanced scheduler with the library defaults for the kernel that
    serves `kv_dtype`: returns (S, boundaries np.int32 [V, S+1], work
    np.int32 [V*S*U] in launch order, wave_eff); num_sms=0 asks the device."""
    import numpy as np
    arr = _host_i32(seq_lens)
    V = len(arr)
    assert V == B * num_shards
    cap = V * 64 * (-(-q_len * H // 128))
    bnd_out = (ctypes.c_int32 * (V * 65))()
    work_out = (ctypes.c_int32 * cap)()
    S, n, eff = ctypes.c_int(), ctypes.c_int64(), ctypes.c_float()
    _check(library().mla_plan_sched(B, q_len, H, num_shards, _KV_DTYPE[kv_dtype],
                                    arr, num_sms, max_parts, bnd_out,
                                    ctypes.byref(S), work_out, cap,
                                    ctypes.byref(n), ctypes.byref(eff)))
    bnd = np.frombuffer(bnd_out, dtype=np.int32)[:V * (S.value + 1)]
    work = np.frombuffer(work_out, dtype=np.int32)[:n.value].copy()
    return S.value, bnd.reshape(V, S.value + 1).copy(), work, eff.value


def check_page_table(req_to_token, seq_lens, kv_limit, q_len: int,
                     num_slots: int, page_size: int = PAGE_SIZE) -> None:
    """Host validation of a page table (raises MlaError on a bad entry)."""
    r2t = req_to_token.detach().to("cpu", torch.int32).contiguous()
    sl = seq_lens.detach().to("cpu", torch.int32).contiguous()
    kl = None if kv_limit is None else kv_limit.detach().to("cpu", torch.int32).contiguous()
    _check(library().mla_check_page_table(
        _ptr(r2t), r2t.shape[1], _ptr(sl), _ptr(kl), r2t.shape[0], q_len,
        page_size, num_slots))


# ------------------------------------------------------------------ kernels
def _kv_dtype(kv: torch.Tensor) -> int:
    if kv.dtype == torch.bfloat16:
        return KV_BF16
    if kv.dtype in (torch.uint8, torch.float8_e4m3fn):
        return KV_FP8_E4M3
    raise TypeError(f"kv dtype {kv.dtype}: expected bfloat16 or uint8 (E4M3)")


def decode_partial(q_nope, q_rope, kv, kv_scale, req_to_token, seq_lens,
                   kv_limit, num_splits: int, sm_scale: float,
                   num_shards: int = 1, O_part=None, LSE_part=None,
                   status=None, simt: bool = False, stream=None,
                   split_pages=None, work=None, part_dtype=None):
    """Partial (O, LSE) per split and shard; see mla_decode_partial.
    `split_pages`: device int32 [num_shards*B, num_splits+1] or None;
    `work`: device int32 unit ids in launch order (plan_sched) or None
    (tensor-core path only).  A bf16 O_part (given, or part_dtype=
    torch.bfloat16) calls mla_decode_partial_bf16_parts.

    Returns (O_part [S, shards, B, q, H, 512], fp32 unless bf16 was asked
    for, LSE_part fp32 [S, shards, B, q, H]); outputs are allocated with
    torch unless given.
    """
    B, q_len, H, _ = q_nope.shape
    dev = q_nope.device
    if O_part is None:
        O_part = torch.empty((num_splits, num_shards, B, q_len, H, VALUE_DIM),
                             dtype=part_dtype or torch.float32, device=dev)
    bf16_parts = O_part.dtype == torch.bfloat16
    if LSE_part is None:
        LSE_part = torch.empty((num_splits, num_shards, B, q_len, H),
                               dtype=torch.float32, device=dev)
    args = (_ptr(q_nope), _ptr(q_rope), _ptr(kv), _ptr(kv_scale),
            _kv_dtype(kv), kv.shape[0], _ptr(req_to_token),
            req_to_token.stride(0), _ptr(seq_lens), _ptr(kv_limit), B, q_len,
            H, num_shards, PAGE_SIZE, float(sm_scale), num_splits,
            _ptr(split_pages))
    with _on(q_nope):
        tail = (_ptr(O_part), _ptr(LSE_part), _ptr(status), _stream(stream))
        if simt:
            if work is not None or bf16_parts:
                raise ValueError("the CUDA-core path takes no work list and "
                                 "writes fp32 parts")
            _check(library().mla_decode_partial_simt(*args, *tail))
        else:
            fn = (library().mla_decode_partial_bf16_parts if bf16_parts
                  else library().mla_decode_partial)
            _check(fn(*args, _ptr(work), 0 if work is None else work.numel(), *tail))
    return O_part, LSE_part


def fused_counters(B: int, q_len: int, H: int, device) -> torch.Tensor:
    """Zeroed arrival counters for decode_fused (int32 [B * ceil(q_len*H/128)]);
    every call leaves them zero again, so one tensor serves every call."""
    return torch.zeros((B * ((q_len * H + 127) // 128),), dtype=torch.int32,
                       device=device)


def decode_fused(q_nope, q_rope, kv, kv_scale, req_to_token, seq_lens,
                 kv_limit, num_splits: int, sm_scale: float,
                 num_shards: int = 1, O_part=None, LSE_part=None,
                 counters=None, out=None, lse_out=None, status=None,
                 stream=None, split_pages=None, work=None):
    """Partial decode and LSE combine in one launch; see mla_decode.

    Returns (out bf16 [B, q, H, 512], lse fp32 [B, q, H]); workspace and
    outputs are allocated with torch unless given."""
    B, q_len, H, _ = q_nope.shape
    dev = q_nope.device
    if O_part is None:
        O_part = torch.empty((num_splits, num_shards, B, q_len, H, VALUE_DIM),
                             dtype=torch.float32, device=dev)
    if LSE_part is None:
        LSE_part = torch.empty((num_splits, num_shards, B, q_len, H),
                               dtype=torch.float32, device=dev)
    if counters is None:
        counters = fused_counters(B, q_len, H, dev)
    if out is None:
        out = torch.empty((B, q_len, H, VALUE_DIM), dtype=torch.bfloat16, device=dev)
    if lse_out is None:
        lse_out = torch.empty((B, q_len, H), dtype=torch.float32, device=dev)
    with _on(q_nope):
        _check(library().mla_decode(
            _ptr(q_nope), _ptr(q_rope), _ptr(kv), _ptr(kv_scale), _kv_dtype(kv),
            kv.shape[0], _ptr(req_to_token), req_to_token.stride(0),
            _ptr(seq_lens), _ptr(kv_limit), B, q_len, H, num_shards, PAGE_SIZE,
            float(sm_scale), num_splits, _ptr(split_pages), _ptr(work),
            0 if work is None else work.numel(), _ptr(O_part), _ptr(LSE_part),
            _ptr(counters), _ptr(out), _ptr(lse_out), _ptr(status),
            _stream(stream)))
    return out, lse_out


def scratch_bytes(B: int, q_len: int, H: int, num_shards: int,
                  num_splits: int) -> int:
    """Static scratch bytes decode_scratch needs (see mla_scratch_bytes)."""
    return _check(library().mla_scratch_bytes(B, q_len, H, num_shards, num_splits))


def decode_scratch(q_nope, q_rope, kv, kv_scale, req_to_token, seq_lens,
                   kv_limit, num_splits: int, sm_scale: float,
                   num_shards: int = 1, out=None, lse_out=None, status=None,
                   stream=None, split_pages=None, work=None):
    """decode_fused with its workspace in the library's static scratch; see
    mla_decode_scratch (calls that may overlap on a device race on it)."""
    B, q_len, H, _ = q_nope.shape
    dev = q_nope.device
    if out is None:
        out = torch.empty((B, q_len, H, VALUE_DIM), dtype=torch.bfloat16, device=dev)
    if lse_out is None:
        lse_out = torch.empty((B, q_len, H), dtype=torch.float32, device=dev)
    with _on(q_nope):  # the scratch array used is the current device's
        _check(library().mla_decode_scratch(
            _ptr(q_nope), _ptr(q_rope), _ptr(kv), _ptr(kv_scale), _kv_dtype(kv),
            kv.shape[0], _ptr(req_to_token), req_to_token.stride(0),
            _ptr(seq_lens), _ptr(kv_limit), B, q_len, H, num_shards, PAGE_SIZE,
            float(sm_scale), num_splits, _ptr(split_pages), _ptr(work),
            0 if work is None else work.numel(), _ptr(out), _ptr(lse_out),
            _ptr(status), _stream(stream)))
    return out, lse_out


def kv_write(rows, slots, kv, kv_scale=None, status=None, stream=None):
    """Store bf16 latent rows [n, 576] at `slots` of the pool `kv` (bf16, or
    uint8 E4M3 bytes with `kv_scale`); see mla_kv_write."""
    n = rows.shape[0]
    _check(library().mla_kv_write(_ptr(rows), n, _ptr(slots), _ptr(kv),
                                  _kv_dtype(kv), _ptr(kv_scale), kv.shape[0],
                                  _ptr(status), _stream(stream)))


def absorb_q(q_nope, w_kc, out=None, status=None, stream=None):
    """q_nope bf16 [B, q, H, 128] . w_kc bf16 [H, 128, 512] -> bf16 [B, q, H,
    512] (the absorbed query); see mla_absorb_q."""
    B, q, H, _ = q_nope.shape
    if out is None:
        out = torch.empty((B, q, H, NOPE_DIM), dtype=torch.bfloat16, device=q_nope.device)
    _check(library().mla_absorb_q(_ptr(q_nope), _ptr(w_kc), _ptr(out), B * q, H,
                                  _ptr(status), _stream(stream)))
    return out


def project_out(o_latent, w_vc, out=None, status=None, stream=None):
    """o_latent bf16 [B, q, H, 512] . w_vc bf16 [H, 512, 128] -> bf16 [B, q, H,
    128]; see mla_project_out."""
    B, q, H, _ = o_latent.shape
    if out is None:
        out = torch.empty((B, q, H, 128), dtype=torch.bfloat16, device=o_latent.device)
    _check(library().mla_project_out(_ptr(o_latent), _ptr(w_vc), _ptr(out), B * q,
                                     H, _ptr(status), _stream(stream)))
    return out


def lse_combine(O_part, LSE_part, out=None, lse_out=None, stream=None):
    """LSE merge over the leading part dims -> (bf16 [rows, 512], fp32 [rows])."""
    value_shape = LSE_part.shape
    nd = LSE_part.dim()
    parts = 1
    # leading dims (splits, shards) are parts; the rest are rows
    lead = 2 if nd == 5 else 1
    for d in value_shape[:lead]:
        parts *= d
    rows = LSE_part.numel() // parts
    row_shape = tuple(value_shape[lead:])
    if out is None:
        out = torch.empty(row_shape + (VALUE_DIM,), dtype=torch.bfloat16,
                          device=O_part.device)
    if lse_out is None:
        lse_out = torch.empty(row_shape, dtype=torch.float32, device=O_part.device)
    fn = (library().mla_lse_combine_bf16_parts if O_part.dtype == torch.bfloat16
          else library().mla_lse_combine)
    _check(fn(_ptr(O_part), _ptr(LSE_part), parts, rows, _ptr(out), _ptr(lse_out),
              _stream(stream)))
    return out, lse_out


def debug_gather(kv, req_to_token, seq_lens, row_offset, total_rows: int,
                 stream=None):
    """Raw-byte gather of every live token row through the TMA path."""
    out = torch.empty((max(total_rows, 1), ROW_DIM), dtype=kv.dtype, device=kv.device)
    _check(library().mla_debug_gather(
        _ptr(kv), _kv_dtype(kv), kv.shape[0], _ptr(req_to_token),
        req_to_token.stride(0), _ptr(seq_lens), _ptr(row_offset),
        req_to_token.shape[0], PAGE_SIZE, _ptr(out), _stream(stream)))
    return out[:total_rows]


def debug_wait(mode: int, delay_us: int, status, elapsed_ns, stream=None):
    """Run the kernels' bounded wait on a barrier phase that nothing
    completes (mode 0), that another warp aborts (1) or completes (2) after
    delay_us; see mla_debug_wait.  `status` int32 [1], `elapsed_ns` int64 [1]
    (device)."""
    with _on(status):
        _check(library().mla_debug_wait(mode, delay_us, _ptr(status),
                                        _ptr(elapsed_ns), _stream(stream)))


def debug_quotients(counters, stream=None):
    """Exhaustive check of the FP8 cache write's division routine against the
    IEEE division (see mla_debug_quotients); `counters` int64 [2] on the
    device, zeroed: bit mismatches, code mismatches are added."""
    with _on(counters):
        _check(library().mla_debug_quotients(
            ctypes.c_void_p(counters.data_ptr()),
            ctypes.c_void_p(counters.data_ptr() + 8), _stream(stream)))


def decode(batch, num_splits: Optional[int] = None, simt: bool = False,
           status=None, stream=None, split_pages=None, fused: bool = False,
           work=None):
    """One decode step of a synth.Batch-like object: partial + combine (two
    launches, or one with fused=True).

    Without num_splits the work-balanced scheduler chooses the parts and the
    launch order (mla_plan_sched; the CUDA-core path takes the parts only);
    with num_splits and no split_pages the pages are dealt uniformly.
    Returns (out bf16 [B, q, H, 512], lse fp32 [B, q, H], num_splits).

    Planning reads the lengths back from the device and uploads the plan
    synchronously, so the host waits for earlier work on the stream.  A
    serving loop keeps the lengths on the host and calls plan_sched,
    decode_partial and lse_combine itself, with the plan uploaded from pinned
    memory on its own stream (bench.py's end-to-end loop does that).
    """
    wl = batch.wl
    if num_splits is None and wl.num_splits:
        num_splits = wl.num_splits
    if num_splits is None:
        num_splits, bnd, wk, _ = plan_sched(
            wl.B, wl.q_len, wl.H, batch_lengths(batch), wl.num_shards,
            kv_dtype=wl.kv_dtype)
        split_pages = torch.from_numpy(bnd).to(batch.q_nope.device)
        if not simt:
            work = torch.from_numpy(wk).to(batch.q_nope.device)
    if fused:
        out, lse = decode_fused(
            batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
            batch.req_to_token, batch.seq_lens, batch.kv_limit, num_splits,
            wl.sm_scale, num_shards=wl.num_shards, status=status, stream=stream,
            split_pages=split_pages, work=work)
        return out, lse, num_splits
    O_part, LSE_part = decode_partial(
        batch.q_nope, batch.q_rope, batch.kv, batch.kv_scale,
        batch.req_to_token, batch.seq_lens, batch.kv_limit, num_splits,
        wl.sm_scale, num_shards=wl.num_shards, status=status, simt=simt,
        stream=stream, split_pages=split_pages, work=work)
    out, lse = lse_combine(O_part, LSE_part, stream=stream)
    return out, lse, num_splits


def batch_lengths(batch):
    """Host list of the (virtual) request lengths of a batch."""
    return [int(x) for x in batch.seq_lens.tolist()]
