"""Shared helpers of the GPU parity tests: oracle calls and tolerance checks.

Tolerances follow the stated bar for GPU vs oracle: BF16 KV max-abs 2e-2 and
relative L2 1e-2; FP8 KV 5e-2 and 2e-2; LSE within 1e-3 absolute.
"""
import math

import numpy as np
import torch

import oracle
from mla_latent_decode_gb300 import synth

TOL = {"bf16": (2e-2, 1e-2), "fp8_e4m3": (5e-2, 2e-2)}
LSE_TOL = 1e-3


def oracle_rows(batch, hb, rows, shard=None, lo=None, hi=None):
    """Oracle O/LSE for flat rows of the [B, q, H] layout (optionally of one
    context shard, optionally over a token range)."""
    wl = batch.wl
    B = wl.B
    r2t, sl, kl = hb["req_to_token"], hb["seq_lens"], hb["kv_limit"]
    if shard is not None:
        r2t = r2t[shard * B:(shard + 1) * B]
        sl = sl[shard * B:(shard + 1) * B]
        kl = None if kl is None else kl[shard * B:(shard + 1) * B]
    return oracle.mla_decode_rows(hb["q_nope"], hb["q_rope"], hb["kv"], batch.kv_is_fp8,
                                  hb["kv_scale"], r2t, sl, kl, B, wl.q_len, wl.H,
                                  wl.sm_scale, rows, lo, hi)


def compact_unsharded(batch, reqs):
    """Host oracle inputs for requests `reqs` of a (possibly sharded) batch,
    unsharded: each request's tokens in logical order (token p of request b
    is local token p // S of shard p % S, the interleaving of the pages'
    context-parallel layout), gathered from the very bytes the kernel reads
    into a compact pool.  Returns (host dict for oracle.mla_decode_rows,
    B' = len(reqs))."""
    wl = batch.wl
    S, B = wl.num_shards, wl.B
    dev = batch.kv.device
    rows, scales, lens = [], [], []
    for b in reqs:
        L = wl.seq_lens[b]
        p = torch.arange(L, device=dev, dtype=torch.int64)
        if S == 1:
            slots = batch.req_to_token[b, p]
        else:
            slots = batch.req_to_token[(p % S) * B + b, p // S]
        slots = slots.to(torch.int64)
        rows.append(batch.kv.index_select(0, slots))
        if batch.kv_is_fp8:
            scales.append(batch.kv_scale.index_select(0, slots))
        lens.append(L)
    pool = torch.cat(rows)
    stride = max(lens)
    r2t = np.zeros((len(reqs), stride), np.int32)
    off = 0
    for i, L in enumerate(lens):
        r2t[i, :L] = off + np.arange(L, dtype=np.int32)
        off += L
    idx = torch.tensor(reqs, device=batch.q_nope.device)

    def bits16(t):
        return t.contiguous().view(torch.int16).cpu().numpy().view("uint16")
    host = dict(q_nope=bits16(batch.q_nope.index_select(0, idx)),
                q_rope=bits16(batch.q_rope.index_select(0, idx)),
                req_to_token=r2t, seq_lens=np.array(lens, np.int32),
                kv_limit=None)
    if batch.kv_is_fp8:
        host["kv"] = pool.cpu().numpy()
        host["kv_scale"] = torch.cat(scales).cpu().numpy()
    else:
        host["kv"] = bits16(pool)
        host["kv_scale"] = None
    return host, len(reqs)


def oracle_rows_host(host, Bq, wl, kv_is_fp8, rows):
    """Oracle O/LSE for flat rows of the [Bq, q, H] layout of a host dict."""
    return oracle.mla_decode_rows(host["q_nope"], host["q_rope"], host["kv"],
                                  kv_is_fp8, host["kv_scale"],
                                  host["req_to_token"], host["seq_lens"], None,
                                  Bq, wl.q_len, wl.H, wl.sm_scale, rows)


def split_range(L, S, s, page=64):
    P = -(-L // page)
    return (s * P // S) * page, min(((s + 1) * P // S) * page, L)


def check_close(got_O, got_lse, ref_O, ref_lse, kv_dtype, what=""):
    """Element-by-element comparison under the stated tolerances."""
    got_O = np.asarray(got_O, np.float64)
    ref_O = np.asarray(ref_O, np.float64)
    got_lse = np.asarray(got_lse, np.float64)
    ref_lse = np.asarray(ref_lse, np.float64)
    max_abs_tol, rel_tol = TOL[kv_dtype]
    assert np.isfinite(got_O).all(), f"{what}: non-finite O"
    err = np.abs(got_O - ref_O)
    max_abs = float(err.max()) if err.size else 0.0
    rel = float(np.linalg.norm(got_O - ref_O) / max(np.linalg.norm(ref_O), 1e-30))
    assert max_abs <= max_abs_tol, f"{what}: max-abs {max_abs:.3e} > {max_abs_tol}"
    assert rel <= rel_tol, f"{what}: rel-L2 {rel:.3e} > {rel_tol}"
    both_inf = np.isneginf(got_lse) & np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse)), f"{what}: empty rows differ"
    dl = np.abs(got_lse[~both_inf] - ref_lse[~both_inf])
    max_dl = float(dl.max()) if dl.size else 0.0
    assert max_dl <= LSE_TOL, f"{what}: LSE err {max_dl:.3e} > {LSE_TOL}"
    return dict(max_abs=max_abs, rel_l2=rel, lse=max_dl)


def f64(t):
    return t.detach().to(torch.float64).cpu().numpy()
