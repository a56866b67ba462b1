"""Seeded synthetic inputs for DSA sparse MLA.

This module only draws random numbers and lays them out in memory; it holds
none of the method's arithmetic (no top-k, no attention, no combine).  The
CUDA path and the fp64 oracle both consume what it produces, so parity is
always checked on identical inputs.

Workload shapes follow the GLM-5.3-Flash serving pages ("Accelerating
GLM-5.3-Flash on H200", section 1 "Architecture and workloads": 64K-token
contexts, 99.9% shared prefix for decode; section 3: 8-token speculative
verify; the vLLM PCP/DCP digest: 1M-token contexts; the SGLang cookbook: FP8
E4M3 KV on Blackwell).  Layout of a KV row: latent || rope as FP8 E4M3 bytes,
one fp32 scale per token (max-abs / 448).  Prefix pages are shared between
requests the way a KV-only RadixCache shares them (section 2, "KV-only decode
RadixCache"): N requests with prefix Lp and suffix Ls occupy Lp + N*Ls token
slots, plus the page-alignment overhead that the page ignores.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

E4M3_MAX = 448.0


@dataclass(frozen=True)
class Workload:
    name: str
    num_req: int
    q_per_req: int
    heads: int
    d_latent: int
    d_rope: int
    ctx: int  # KV positions per request, including the query tokens' own rows
    shared_prefix: int  # Lp: tokens shared by all requests (before page alignment)
    page_size: int
    k: int
    seed: int
    softmax_scale: float | None = None  # default 1/sqrt(d_latent + d_rope)
    tie_frac: float = 0.0  # per row, this fraction of visible positions copies another's score
    spike_frac: float = 0.0  # per row, this fraction of positions is replaced by Laplace spikes
    spike_scale: float = 5.0
    ctx_per_req: tuple | None = None  # ragged contexts (default: every request has ctx)
    share_pages: bool = True  # False: every request keeps its own copy of the prefix pages

    @property
    def dqk(self) -> int:
        return self.d_latent + self.d_rope

    @property
    def num_q(self) -> int:
        return self.num_req * self.q_per_req

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale is not None else 1.0 / math.sqrt(self.dqk)

    def contexts(self) -> list[int]:
        if self.ctx_per_req is not None:
            assert len(self.ctx_per_req) == self.num_req
            return [int(c) for c in self.ctx_per_req]
        return [self.ctx] * self.num_req

    @property
    def ld_scores(self) -> int:
        return max(self.contexts())


# The five workloads the path is measured and checked on.
TINY = Workload("tiny_decode_h16_ctx512", 2, 1, 16, 64, 16, 512, 256, 16, 64, seed=0,
                softmax_scale=1.0 / math.sqrt(80.0), tie_frac=0.05)
DECODE_64K = Workload("decode_64k_prefix99.9", 128, 1, 64, 512, 64, 65536, 65470, 64, 2048, seed=1)
VERIFY_64K = Workload("verify_64k_8tok", 128, 8, 64, 512, 64, 65536, 0, 64, 2048, seed=2)
PREFILL_32K = Workload("prefill_32k_on_32k", 1, 32768, 64, 512, 64, 65536, 0, 64, 2048, seed=3)
CTX_1M = Workload("ctx_1m_4x4", 4, 4, 64, 512, 64, 1 << 20, 0, 64, 2048, seed=4, spike_frac=0.001)
WORKLOADS = {w.name: w for w in (TINY, DECODE_64K, VERIFY_64K, PREFILL_32K, CTX_1M)}

# Smaller cases of the same kernels for profiler captures (a few hundred MB on
# the device): the verify block with 19 requests, 152 query tokens, one
# attention CTA per SM, its pool (717 MB) still far larger than L2.
VERIFY_64K_ONE_WAVE = replace(VERIFY_64K, name="verify_64k_8tok_19req", num_req=19)
PROFILE_CASES = {w.name: w for w in (VERIFY_64K_ONE_WAVE,)}


def lookup(name: str) -> Workload:
    """A measured workload, else a profiling case, by name."""
    return WORKLOADS[name] if name in WORKLOADS else PROFILE_CASES[name]


def shrink(w: Workload, **kw) -> Workload:
    return replace(w, **kw)


@dataclass
class PageLayout:
    block_table: torch.Tensor  # int32 [num_req, max_pages]; -1 past a request's last page
    num_pages: int
    n_shared_pages: int



def page_layout(w: Workload, gen: torch.Generator, device) -> PageLayout:
    """Block tables.  Whole pages of the shared prefix get ids 0..n-1 and are
    referenced by every request; a prefix tail shorter than a page is copied
    into each request's first private page.  Private page ids are a seeded
    permutation of the remaining ids, handed out request by request, so the
    gathers are genuinely indirect."""
    P = w.page_size
    ctxs = w.contexts()
    n_shared = (w.shared_prefix // P) if w.share_pages else 0
    pages_per_req = [math.ceil(c / P) for c in ctxs]
    assert all(p >= n_shared for p in pages_per_req)
    n_private = sum(p - n_shared for p in pages_per_req)
    total = n_shared + n_private
    perm = torch.randperm(n_private, generator=gen, device=gen.device).to(torch.int32) + n_shared
    max_pages = max(pages_per_req)
    bt = torch.full((w.num_req, max_pages), -1, dtype=torch.int32, device=gen.device)
    off = 0
    for r, npg in enumerate(pages_per_req):
        if n_shared:
            bt[r, :n_shared] = torch.arange(n_shared, dtype=torch.int32, device=gen.device)
        m = npg - n_shared
        bt[r, n_shared:npg] = perm[off:off + m]
        off += m
    return PageLayout(bt.to(device), total, n_shared)


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + stream)
    return g


def quantize_rows(x: torch.Tensor):
    """Per-row FP8 E4M3 encoding of fp32 rows: scale = max|row| / 448 and
    bytes = round-to-nearest-even(row / scale), saturated to +-448."""
    amax = x.abs().amax(dim=1).clamp_min(1e-30)
    scale = (amax / E4M3_MAX).to(torch.float32)
    y = (x / scale[:, None]).clamp(-E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn).view(torch.uint8), scale


def _randn_rows(n: int, d: int, g: torch.Generator, device) -> torch.Tensor:
    return torch.randn((n, d), generator=g, device=device, dtype=torch.float32)


@dataclass
class Inputs:
    w: Workload
    q: torch.Tensor  # bf16 [num_q, H, dqk]
    kv: torch.Tensor  # uint8 (e4m3 bits) [slots, dqk]
    kv_scale: torch.Tensor  # fp32 [slots]
    block_table: torch.Tensor  # int32 [num_req, max_pages]
    q_pos: torch.Tensor  # int32 [num_q]
    q_req: torch.Tensor  # int32 [num_q]
    scores: torch.Tensor  # fp32 [num_q, ld_scores]
    layout: PageLayout
    logical: list | None = None  # per request: (uint8 [ctx, dqk], fp32 [ctx]) in position order

    @property
    def num_pages(self) -> int:
        return self.layout.num_pages


def make_inputs(w: Workload, device="cpu", row_chunk: int = 1 << 18, with_scores: bool = True,
                keep_logical: bool = False) -> Inputs:
    """All inputs of one workload on ``device``.  With ``keep_logical`` the
    result also carries each request's rows in position order (bytes, scales),
    independent of the page layout (for small checks only)."""
    device = torch.device(device)
    P, dqk = w.page_size, w.dqk
    ctxs = w.contexts()
    layout = page_layout(w, _gen(w.seed, 1, device), device)
    slots = layout.num_pages * P
    kv = torch.zeros((slots, dqk), dtype=torch.uint8, device=device)
    kv_scale = torch.ones((slots,), dtype=torch.float32, device=device)
    bt = layout.block_table

    g_kv = _gen(w.seed, 2, device)
    Lp = w.shared_prefix
    prefix_bytes = prefix_scale = None
    if Lp > 0:
        prefix_bytes, prefix_scale = quantize_rows(_randn_rows(Lp, dqk, g_kv, device))
    n_shared_tok = layout.n_shared_pages * P
    logical = [] if keep_logical else None

    def put(r, lo, hi, b, s):
        pos = torch.arange(lo, hi, device=device, dtype=torch.int64)
        slot = bt[r].to(torch.int64)[pos // P] * P + pos % P
        kv[slot] = b
        kv_scale[slot] = s

    for r, c in enumerate(ctxs):
        parts_b, parts_s = [], []
        if Lp > 0:
            # whole shared pages are written once (by request 0); a copy of the
            # prefix tail (and, without sharing, of the whole prefix) goes into
            # each request's private pages
            p_lo = 0 if r == 0 else n_shared_tok
            if p_lo < Lp:
                put(r, p_lo, Lp, prefix_bytes[p_lo:Lp], prefix_scale[p_lo:Lp])
            if logical is not None:
                parts_b.append(prefix_bytes)
                parts_s.append(prefix_scale)
        for lo in range(Lp, c, row_chunk):
            hi = min(c, lo + row_chunk)
            b, s = quantize_rows(_randn_rows(hi - lo, dqk, g_kv, device))
            put(r, lo, hi, b, s)
            if logical is not None:
                parts_b.append(b)
                parts_s.append(s)
        if logical is not None:
            logical.append((torch.cat(parts_b), torch.cat(parts_s)))

    q_pos = torch.cat([torch.arange(c - w.q_per_req, c, dtype=torch.int32) for c in ctxs]).to(device)
    q_req = torch.arange(w.num_req, dtype=torch.int32).repeat_interleave(w.q_per_req).to(device)
    g_q = _gen(w.seed, 3, device)
    q = torch.randn((w.num_q, w.heads, dqk), generator=g_q, device=device, dtype=torch.float32).to(torch.bfloat16)

    scores = torch.empty(0, dtype=torch.float32, device=device)
    if with_scores:
        scores = make_scores(w, q_pos, device)
    return Inputs(w, q, kv, kv_scale, bt, q_pos, q_req, scores, layout, logical)


def make_scores(w: Workload, q_pos: torch.Tensor, device) -> torch.Tensor:
    """fp32 indexer scores N(0,1) [num_q, ld].  Optional exact ties: per row,
    floor(tie_frac * visible) visible positions (without replacement) copy the
    score of another uniformly drawn visible position.  Optional spikes: per
    row, floor(spike_frac * ld) visible positions (without replacement) are
    replaced by Laplace(0, spike_scale) draws."""
    device = torch.device(device)
    ld = w.ld_scores
    g = _gen(w.seed, 4, device)
    scores = torch.randn((w.num_q, ld), generator=g, device=device, dtype=torch.float32)
    if w.tie_frac > 0 or w.spike_frac > 0:
        qp = q_pos.cpu().tolist()
        g2 = _gen(w.seed, 5, device)
        for i, p in enumerate(qp):
            vis = p + 1
            if w.tie_frac > 0 and vis > 1:
                nt = int(math.floor(w.tie_frac * vis))
                dst = torch.randperm(vis, generator=g2, device=device)[:nt]
                off = torch.randint(1, vis, (nt,), generator=g2, device=device)
                src = (dst + off) % vis
                row = scores[i]
                row[dst] = row[src].clone()
            if w.spike_frac > 0:
                ns = int(math.floor(w.spike_frac * ld))
                dst = torch.randperm(vis, generator=g2, device=device)[:ns]
                u = torch.rand((ns,), generator=g2, device=device, dtype=torch.float64) - 0.5
                lap = -w.spike_scale * torch.sign(u) * torch.log1p(-2.0 * u.abs())
                scores[i, dst] = lap.to(torch.float32)
    return scores


def slot_count(w: Workload) -> int:
    """Token slots the layout occupies: whole shared prefix pages once, plus
    each request's private pages (prefix tail copy + suffix)."""
    P = w.page_size
    n_shared = (w.shared_prefix // P) if w.share_pages else 0
    return P * (n_shared + sum(math.ceil(c / P) - n_shared for c in w.contexts()))
