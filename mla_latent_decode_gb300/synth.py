"""Seeded synthetic inputs with the shapes of the pages' decode workloads.

This module only draws random numbers and lays them out in the paged latent
KV format; it contains none of the attention arithmetic.  Both the CUDA path
(through ``bench.py`` and the tests) and the CPU oracle consume what it makes.

Layout (the pages' SGLang-style pool, see "Resident VRAM: weights and KV
cache", sections on cell_size and req_to_token):
  * ``kv``: one latent row per slot, ``[num_slots, 576]`` = c_kv (512) then
    the RoPE key (64), BF16, or OCP E4M3 bytes plus one fp32 scale per slot.
  * slots come in pages of 64; page 0 is a dummy page.  Each request owns a
    random permutation of pages; ``req_to_token[b, t]`` is the slot of token
    ``t`` (every token has an entry; the pages are contiguous runs of 64).
  * slots that hold no token (the dummy page, the tail of a request's last
    page) are filled with NaN so that any leak shows up.

Seeds (sub-streams of one seed s): queries s, KV s+1, page permutation s+2,
sequence lengths s+3.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

ROW_DIM, NOPE_DIM, ROPE_DIM, VALUE_DIM = 576, 512, 64, 512
PAGE_SIZE = 64
BF16_NAN_BITS = 0x7FC0
E4M3_NAN_BYTE = 0x7F
E4M3_MAX = 448.0


@dataclass
class Workload:
    """One decode-step workload: shapes, lengths and the KV storage type."""

    name: str
    B: int
    q_len: int
    H: int
    seq_lens: List[int]
    kv_dtype: str = "bf16"          # "bf16" | "fp8_e4m3"
    sm_scale: float = 1.0 / math.sqrt(192.0)
    page_size: int = PAGE_SIZE
    num_shards: int = 1             # token-interleaved context shards
    q_scale: float = 1.0            # >1 gives a peaked softmax
    num_splits: Optional[int] = None  # None: use the wave-rounding planner

    @property
    def rows(self) -> int:
        return self.B * self.q_len * self.H

    def flops(self) -> int:
        """Algorithmic FLOPs: 2*(576+512) per (query row, visible token)."""
        vis = 0
        for L in self.seq_lens:
            for i in range(self.q_len):
                vis += L - self.q_len + 1 + i
        return 2 * self.H * (ROW_DIM + VALUE_DIM) * vis

    def kv_row_bytes(self) -> int:
        return ROW_DIM * 2 if self.kv_dtype == "bf16" else ROW_DIM + 4


def _ragged_lengths(B: int, lo: int, hi: int, seed: int) -> List[int]:
    g = torch.Generator().manual_seed(seed + 3)
    u = torch.rand(B, generator=g, dtype=torch.float64)
    lens = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    return [int(round(float(x))) for x in lens]


def config(name: str, seed: int = 0, **over) -> Workload:
    """The named decode workloads.

    tiny        1 request, q_len 1, 16 heads, 256-token context, BF16, 1 split
    dp16        16 requests x q_len 5 x 96 heads x 100k context, BF16
    dcp         128 requests x q_len 5 x 96 heads x 100k context split into 8
                token-interleaved shards (~12.5k tokens each), BF16
    ragged_fp8  24 requests x q_len 5 x 96 heads, context log-uniform in
                [1k, 200k], FP8 E4M3 KV with a per-token fp32 scale
    sweep_B<b>_L<l>  b requests x q_len 5 x 96 heads x l context, BF16
    sweep8_B<b>_L<l> the same with FP8 E4M3 KV and a per-token fp32 scale
    dcp_B<b>    b requests of dcp's shape (8 shards of 100k tokens): a
                smaller case of the same kernel launch
    """
    if name == "tiny":
        wl = Workload("tiny", 1, 1, 16, [256], num_splits=1)
    elif name == "dp16":
        wl = Workload("dp16", 16, 5, 96, [100_000] * 16)
    elif name == "dcp":
        wl = Workload("dcp", 128, 5, 96, [100_000] * 128, num_shards=8)
    elif name == "ragged_fp8":
        wl = Workload("ragged_fp8", 24, 5, 96,
                      _ragged_lengths(24, 1_000, 200_000, seed), "fp8_e4m3")
    elif name.startswith("sweep_B"):
        b, l = name[len("sweep_B"):].split("_L")
        wl = Workload(name, int(b), 5, 96, [int(l)] * int(b))
    elif name.startswith("dcp_B"):
        b = int(name[len("dcp_B"):])
        wl = Workload(name, b, 5, 96, [100_000] * b, num_shards=8)
    elif name.startswith("sweep8_B"):
        b, l = name[len("sweep8_B"):].split("_L")
        wl = Workload(name, int(b), 5, 96, [int(l)] * int(b), "fp8_e4m3")
    else:
        raise KeyError(name)
    for k, v in over.items():
        setattr(wl, k, v)
    return wl


@dataclass
class Batch:
    """Device (or host) tensors of one workload, in the kernel's layout.

    With ``num_shards`` = S > 1 the KV tables describe S*B virtual requests,
    v = shard * B + b, each holding the positions p = shard (mod S) of request b
    in ascending order; ``kv_limit`` then gives each query's visible count.
    """

    wl: Workload
    q_nope: torch.Tensor            # bf16 [B, q_len, H, 512]
    q_rope: torch.Tensor            # bf16 [B, q_len, H, 64]
    kv: torch.Tensor                # bf16 or uint8 [num_slots, 576]
    kv_scale: Optional[torch.Tensor]  # fp32 [num_slots] (FP8 only)
    req_to_token: torch.Tensor      # int32 [S*B, stride]
    seq_lens: torch.Tensor          # int32 [S*B]
    kv_limit: Optional[torch.Tensor]  # int32 [S*B, q_len] or None
    page_tables: List[torch.Tensor] = field(default_factory=list)

    @property
    def num_slots(self) -> int:
        return int(self.kv.shape[0])

    @property
    def kv_is_fp8(self) -> bool:
        return self.wl.kv_dtype != "bf16"


def shard_lengths(L: int, q_len: int, S: int, s: int):
    """Local length and per-query visible counts of shard s of a request.

    Shard s holds positions p = s, s+S, s+2S, ... < L; query i sees
    positions p <= L - q_len + i, i.e. the first floor((L-q_len+i-s)/S)+1 of
    them (0 if that position precedes s).
    """
    local = 0 if L <= s else (L - s + S - 1) // S
    lim = []
    for i in range(q_len):
        last = L - q_len + i
        lim.append(0 if last < s else (last - s) // S + 1)
    return local, lim


def _fill_pool(num_slots: int, fp8: bool, device) -> torch.Tensor:
    if fp8:
        return torch.full((num_slots, ROW_DIM), E4M3_NAN_BYTE, dtype=torch.uint8,
                          device=device)
    return torch.full((num_slots, ROW_DIM), BF16_NAN_BITS, dtype=torch.int16,
                      device=device).view(torch.bfloat16)


def quantize_e4m3(rows: torch.Tensor):
    """Per-row E4M3 quantiser used to make FP8 test data.

    scale = amax(|row|) / 448; bytes = RNE(row / scale) (saturated to +-448).
    Only the stored bytes and scale define the FP8 workload.
    """
    amax = rows.abs().amax(dim=1).clamp_min(1e-30)
    scale = (amax / E4M3_MAX).to(torch.float32)
    qv = (rows / scale[:, None]).clamp(-E4M3_MAX, E4M3_MAX)
    return qv.to(torch.float8_e4m3fn).view(torch.uint8), scale


def make_batch(wl: Workload, seed: int = 0, device="cpu",
               page_seed: Optional[int] = None, chunk_tokens: int = 1 << 20,
               nan_fill: bool = True) -> Batch:
    """Build the paged inputs of ``wl`` on ``device`` from ``seed``.

    ``page_seed`` overrides the page-permutation stream only, so two batches
    with the same ``seed`` and different ``page_seed`` hold the same logical KV
    under different physical layouts.
    """
    dev = torch.device(device)
    B, q, H, S = wl.B, wl.q_len, wl.H, wl.num_shards
    fp8 = wl.kv_dtype != "bf16"

    gq = torch.Generator(device=dev).manual_seed(seed)
    q_nope = (torch.randn((B, q, H, NOPE_DIM), generator=gq, device=dev,
                          dtype=torch.float32) * wl.q_scale).to(torch.bfloat16)
    q_rope = (torch.randn((B, q, H, ROPE_DIM), generator=gq, device=dev,
                          dtype=torch.float32) * wl.q_scale).to(torch.bfloat16)

    # Virtual requests (shard-major) and their local lengths / limits.
    vlens, vlims = [], []
    for s in range(S):
        for b in range(B):
            if S == 1:
                vlens.append(wl.seq_lens[b])
                vlims.append(None)
            else:
                loc, lim = shard_lengths(wl.seq_lens[b], q, S, s)
                vlens.append(loc)
                vlims.append(lim)
    V = S * B
    ps = wl.page_size
    vpages = [(L + ps - 1) // ps for L in vlens]
    total_pages = sum(vpages)
    num_slots = (1 + total_pages) * ps
    stride = max(1, max(vpages)) * ps

    gp = torch.Generator().manual_seed(seed + 2 if page_seed is None else page_seed)
    perm = (torch.randperm(total_pages, generator=gp) + 1).to(torch.int64)
    r2t = torch.zeros((V, stride), dtype=torch.int32)
    tables, off = [], 0
    for v in range(V):
        pg = perm[off:off + vpages[v]]
        off += vpages[v]
        tables.append(pg)
        if vlens[v]:
            t = torch.arange(vlens[v], dtype=torch.int64)
            r2t[v, :vlens[v]] = (pg[t // ps] * ps + t % ps).to(torch.int32)

    kv = _fill_pool(num_slots, fp8, dev) if nan_fill else (
        torch.zeros((num_slots, ROW_DIM), device=dev,
                    dtype=torch.uint8 if fp8 else torch.bfloat16))
    kv_scale = (torch.full((num_slots,), float("nan"), dtype=torch.float32,
                           device=dev) if fp8 else None)

    # Logical KV rows, request after request in token order, one stream.
    gk = torch.Generator(device=dev).manual_seed(seed + 1)
    r2t_dev = r2t.to(dev)
    for b in range(B):
        L = wl.seq_lens[b]
        for t0 in range(0, L, chunk_tokens):
            n = min(chunk_tokens, L - t0)
            rows = torch.randn((n, ROW_DIM), generator=gk, device=dev,
                               dtype=torch.float32)
            pos = torch.arange(t0, t0 + n, device=dev, dtype=torch.int64)
            if S == 1:
                slots = r2t_dev[b, pos].to(torch.int64)
            else:
                sh = pos % S
                slots = r2t_dev[sh * B + b, pos // S].to(torch.int64)
            if fp8:
                qb, sc = quantize_e4m3(rows)
                kv.index_copy_(0, slots, qb)
                kv_scale.index_copy_(0, slots, sc)
            else:
                kv.index_copy_(0, slots, rows.to(torch.bfloat16))

    seq = torch.tensor(vlens, dtype=torch.int32, device=dev)
    kv_limit = None
    if S > 1:
        kv_limit = torch.tensor(vlims, dtype=torch.int32, device=dev)
    return Batch(wl, q_nope, q_rope, kv, kv_scale, r2t_dev, seq, kv_limit,
                 tables)


def host_bits(batch: Batch) -> dict:
    """Raw storage of a batch as host numpy arrays (bf16 as uint16 bits)."""
    def bits16(t):
        return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")
    d = dict(
        q_nope=bits16(batch.q_nope), q_rope=bits16(batch.q_rope),
        req_to_token=batch.req_to_token.cpu().numpy(),
        seq_lens=batch.seq_lens.cpu().numpy(),
        kv_limit=None if batch.kv_limit is None else batch.kv_limit.cpu().numpy(),
    )
    if batch.kv_is_fp8:
        d["kv"] = batch.kv.cpu().numpy()
        d["kv_scale"] = batch.kv_scale.cpu().numpy()
    else:
        d["kv"] = bits16(batch.kv)
        d["kv_scale"] = None
    return d
