"""Seeded synthetic inputs for the KDA recurrence: the one module that both the CUDA path's
tests/benchmark and the CPU oracle's tests draw from.

It holds no arithmetic of the method: only the input distributions and shapes of the
workloads, and the host-side segment split. Every draw comes from a ``torch.Generator``
seeded per workload, in the fixed order q, k, v, g, beta, initial state (or pool), slots.

Distributions (the workloads' recipe):
  q, v ~ N(0, 1);  k ~ N(0, 1) then L2-normalised over the key channels of each
  (token, head) in fp32, before any cast;  g = -softplus(N(0, 1)) per key channel
  (optionally multiplied by ``decay_scale``; ``decay_scale=0`` gives a = exp(g) = 1 exactly);
  beta = sigmoid(N(0, 1)) (optionally multiplied by ``beta_scale``);  initial states ~ N(0, init_std^2) when requested.
  q, k, v are then rounded to the compute dtype (bf16 with round-to-nearest-even, or kept
  fp32); g, beta and states stay fp32.

Segment leveling follows the split rule of pegainfer pull request #970 ("feat(k3):
cross-process CP whale gang"), whale-rendezvous commit message: segment lengths obey
t ~ len + Q*depth*len with Q = 2.7e-6, so segments that start deeper in the prompt are
shorter, no segment is shorter than the 2048-token floor, and the gang is the widest
power of two that admits that floor (at most 16 members, the widest gang the page runs).
"""
from dataclasses import dataclass, field
from typing import List, Optional

import torch
import torch.nn.functional as F

SEGMENT_FLOOR = 2048
LEVEL_Q = 2.7e-6
MAX_GANG = 16


@dataclass
class PrefillInputs:
    q: torch.Tensor            # [T, H, dk]
    k: torch.Tensor            # [T, H, dk]
    v: torch.Tensor            # [T, H, dv]
    g: torch.Tensor            # [T, H, dk] fp32, <= 0
    beta: torch.Tensor         # [T, H] fp32 in (0, 1)
    cu_seqlens: torch.Tensor   # [N+1] int32
    init_state: Optional[torch.Tensor]  # [N, H, dk, dv] fp32 or None
    lens: List[int] = field(default_factory=list)

    @property
    def T(self):
        return self.k.shape[0]

    @property
    def H(self):
        return self.k.shape[1]

    @property
    def dk(self):
        return self.k.shape[2]

    @property
    def dv(self):
        return self.v.shape[2]


@dataclass
class DecodeInputs:
    q: torch.Tensor          # [B, H, dk]
    k: torch.Tensor          # [B, H, dk]
    v: torch.Tensor          # [B, H, dv]
    g: torch.Tensor          # [B, H, dk] fp32
    beta: torch.Tensor       # [B, H] fp32
    pool: torch.Tensor       # [n_slots, H, dk, dv] fp32
    slot_ids: torch.Tensor   # [B] int32


@dataclass
class WindowInputs:
    q: torch.Tensor            # [B*W, H, dk] (token j of row b is row b*W + j)
    k: torch.Tensor            # [B*W, H, dk]
    v: torch.Tensor            # [B*W, H, dv]
    g: torch.Tensor            # [B*W, H, dk] fp32
    beta: torch.Tensor         # [B*W, H] fp32 in (0, 1)
    beta_logit: torch.Tensor   # [B*W, H] fp32, the N(0, 1) draw that beta is the sigmoid of
    pool: torch.Tensor         # [n_slots, H, dk, dv] fp32
    read_slots: torch.Tensor   # [B] int32
    write_slots: torch.Tensor  # [B, W] int32, disjoint from each other and from read_slots


@dataclass
class ConvInputs:
    x: torch.Tensor            # [T, C] (packed sequences, token-major)
    weight: torch.Tensor       # [C, W] fp32
    cu_seqlens: torch.Tensor   # [N+1] int32
    state: torch.Tensor        # [n_slots, W-1, C], dtype of x
    read_slots: torch.Tensor   # [N] int32
    write_slots: torch.Tensor  # [N] int32, disjoint from read_slots
    lens: List[int] = field(default_factory=list)


_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def _draw_qkvgb(gen, n, H, dk, dv, device, decay_scale, beta_scale=1.0, want_logit=False):
    q = torch.randn(n, H, dk, generator=gen, device=device)
    k = torch.randn(n, H, dk, generator=gen, device=device)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(n, H, dv, generator=gen, device=device)
    g = -F.softplus(torch.randn(n, H, dk, generator=gen, device=device))
    if decay_scale != 1.0:
        g = g * decay_scale
    logit = torch.randn(n, H, generator=gen, device=device)
    beta = torch.sigmoid(logit)
    if beta_scale != 1.0:
        beta = beta * beta_scale
    if want_logit:
        return q, k, v, g, beta, logit
    return q, k, v, g, beta


def make_prefill(lens, H, dk, dv, dtype="bf16", seed=0, device="cpu", init_std=None,
                 decay_scale=1.0, beta_scale=1.0) -> PrefillInputs:
    """Packed sequences of the given lengths (token-major rows, sequences back to back)."""
    lens = [int(x) for x in lens]
    T = sum(lens)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    q, k, v, g, beta = _draw_qkvgb(gen, T, H, dk, dv, device, decay_scale, beta_scale)
    init = None
    if init_std is not None:
        init = torch.randn(len(lens), H, dk, dv, generator=gen, device=device) * init_std
    dt = _DT[dtype]
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return PrefillInputs(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(),
                         v=v.to(dt).contiguous(), g=g.contiguous(), beta=beta.contiguous(),
                         cu_seqlens=cu.to(device), init_state=init, lens=lens)


def make_decode(B, H, dk, dv, n_slots, dtype="bf16", seed=0, device="cpu", pool_std=0.02,
                decay_scale=1.0) -> DecodeInputs:
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    q, k, v, g, beta = _draw_qkvgb(gen, B, H, dk, dv, device, decay_scale)
    pool = torch.randn(n_slots, H, dk, dv, generator=gen, device=device) * pool_std
    slots = torch.randperm(n_slots, generator=gen, device=device)[:B].to(torch.int32)
    dt = _DT[dtype]
    return DecodeInputs(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(),
                        v=v.to(dt).contiguous(), g=g.contiguous(), beta=beta.contiguous(),
                        pool=pool.contiguous(), slot_ids=slots.contiguous())


def make_window(B, W, H, dk, dv, n_slots, dtype="bf16", seed=0, device="cpu", pool_std=0.02,
                decay_scale=1.0) -> WindowInputs:
    """Verify windows: B rows of W tokens each, a pool of n_slots states, and B read slots
    plus B x W write slots sampled without replacement (so every slot is named once)."""
    if B * (W + 1) > n_slots:
        raise ValueError("the pool is too small for distinct read and write slots")
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    q, k, v, g, beta, logit = _draw_qkvgb(gen, B * W, H, dk, dv, device, decay_scale,
                                          want_logit=True)
    pool = torch.randn(n_slots, H, dk, dv, generator=gen, device=device) * pool_std
    perm = torch.randperm(n_slots, generator=gen, device=device)[:B * (W + 1)].to(torch.int32)
    dt = _DT[dtype]
    return WindowInputs(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(),
                        v=v.to(dt).contiguous(), g=g.contiguous(), beta=beta.contiguous(),
                        beta_logit=logit.contiguous(), pool=pool.contiguous(),
                        read_slots=perm[:B].contiguous(),
                        write_slots=perm[B:].reshape(B, W).contiguous())


def make_conv(lens, C, W, dtype="bf16", seed=0, device="cpu", n_slots=None) -> ConvInputs:
    """Short-conv inputs: x ~ N(0, 1) [T, C], weight ~ N(0, 1/W) [C, W], history windows
    ~ N(0, 1) in a pool of n_slots (default 2N) slots, and N read plus N write slots sampled
    without replacement."""
    lens = [int(v) for v in lens]
    N, T = len(lens), sum(lens)
    n_slots = 2 * N if n_slots is None else int(n_slots)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    x = torch.randn(T, C, generator=gen, device=device)
    weight = torch.randn(C, W, generator=gen, device=device) / float(W) ** 0.5
    state = torch.randn(n_slots, max(W - 1, 0), C, generator=gen, device=device)
    perm = torch.randperm(n_slots, generator=gen, device=device)[:2 * N].to(torch.int32)
    cu = torch.zeros(N + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    dt = _DT[dtype]
    return ConvInputs(x=x.to(dt).contiguous(), weight=weight.contiguous(), cu_seqlens=cu.to(device),
                      state=state.to(dt).contiguous(), read_slots=perm[:N].contiguous(),
                      write_slots=perm[N:].contiguous(), lens=lens)


def leveled_split(length, n_segs, q=LEVEL_Q, align=64):
    """Split ``length`` tokens into ``n_segs`` contiguous segments whose lengths satisfy
    len_i * (1 + q * start_i) = tau (deeper segments shorter), each rounded to a multiple of
    ``align``, the last segment taking the remainder. Returns the segment lengths."""
    if n_segs <= 1:
        return [int(length)]

    def lengths_for(tau):
        out, start = [], 0.0
        for _ in range(n_segs):
            ln = tau / (1.0 + q * start)
            out.append(ln)
            start += ln
        return out

    lo, hi = 0.0, float(length) * (1.0 + q * length)
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if sum(lengths_for(mid)) < length:
            lo = mid
        else:
            hi = mid
    raw = lengths_for(0.5 * (lo + hi))
    segs = [int(round(x / align)) * align for x in raw[:-1]]
    segs.append(int(length) - sum(segs))
    return segs


def gang_split(length, floor=SEGMENT_FLOOR, max_gang=MAX_GANG, q=LEVEL_Q, align=64):
    """Widest power-of-two gang (<= max_gang) whose leveled split keeps every segment at or
    above ``floor`` tokens; returns its segment lengths (one segment if none admits)."""
    best = [int(length)]
    p = 2
    while p <= max_gang:
        segs = leveled_split(length, p, q=q, align=align)
        if min(segs) >= floor:
            best = segs
        p *= 2
    return best


def segment_offsets(lens, seg_lens_per_seq):
    """Token offsets [P+1] of all segments (in sequence order) and the per-sequence segment
    offsets [N+1] into that list."""
    offs, seq_seg = [0], [0]
    base = 0
    for ln, segs in zip(lens, seg_lens_per_seq):
        assert sum(segs) == ln
        for s in segs:
            offs.append(offs[-1] + s)
        base += ln
        seq_seg.append(seq_seg[-1] + len(segs))
    return (torch.tensor(offs, dtype=torch.int32), torch.tensor(seq_seg, dtype=torch.int32))


# Strong-coupling variant for the segment path: at the workloads' own decay a 2048-token
# segment's M is exactly zero (the prefix carries no information across it); with the decay
# scaled by 1e-4 and beta by 0.02 the package's M has spectral norm of order one.
STRONG_COUPLING = dict(decay_scale=1e-4, beta_scale=0.02)

# The workloads. Sizes and distributions as stated in each docstring line.
WORKLOADS = {
    # tiny fp32: B=1, H=2, T=256, dk=dv=64, chunk 64, 4 segments of 64, zero init.
    "tiny_fp32": dict(kind="prefill", lens=[256], H=2, dk=64, dv=64, dtype="f32", seed=1000,
                      segs=[[64, 64, 64, 64]]),
    # chunked prefill, one segment: H=32, T=16384, d=128, bf16 q/k/v, zero init.
    "prefill_16k": dict(kind="prefill", lens=[16384], H=32, dk=128, dv=128, dtype="bf16",
                        seed=1001, segs=None),
    # the same inputs split into 8 segments of 2048 tokens.
    "segments_8x2048": dict(kind="prefill", lens=[16384], H=32, dk=128, dv=128, dtype="bf16",
                            seed=1001, segs=[[2048] * 8]),
    # long varlen with nonzero initial states and leveled segments (floor 2048).
    "varlen_long": dict(kind="prefill", lens=[131072, 65536, 32768, 8192], H=32, dk=128,
                        dv=128, dtype="bf16", seed=1003, init_std=0.02, segs="leveled"),
    # decode: 256 sequences x H32 x d128 over a 4096-slot fp32 pool (~8.6 GB).
    "decode_256": dict(kind="decode", B=256, H=32, dk=128, dv=128, n_slots=4096, dtype="bf16",
                       seed=1004, pool_std=0.02),
    # verify windows: 256 rows of 4 tokens (3 drafts + 1 bonus) x H32 x d128 over a 4096-slot
    # pool, each row reading one slot and storing a snapshot per token into 4 others.
    "window_256x4": dict(kind="window", B=256, W=4, H=32, dk=128, dv=128, n_slots=4096,
                         dtype="bf16", seed=1005, pool_std=0.02),
    # short conv over the prefill's q, k and v channels (3 x 32 heads x 128 = 12288 channels)
    # of one 16k-token sequence, width 4, SiLU, history read from one slot, stored to another.
    "conv_16k": dict(kind="conv", lens=[16384], C=12288, W=4, dtype="bf16", seed=1006),
}


def workload_segments(name):
    """Per-sequence segment lengths of a prefill workload (None if it has no split)."""
    w = WORKLOADS[name]
    if w.get("segs") is None:
        return None
    if w["segs"] == "leveled":
        return [gang_split(ln) for ln in w["lens"]]
    return w["segs"]


def make_workload(name, device="cpu", decay_scale=1.0, beta_scale=1.0, **over):
    w = dict(WORKLOADS[name])
    w.update(over)
    if w["kind"] == "conv":
        return make_conv(w["lens"], w["C"], w["W"], w["dtype"], w["seed"], device)
    if w["kind"] == "window":
        return make_window(w["B"], w["W"], w["H"], w["dk"], w["dv"], w["n_slots"], w["dtype"],
                           w["seed"], device, w.get("pool_std", 0.02), decay_scale)
    if w["kind"] == "decode":
        return make_decode(w["B"], w["H"], w["dk"], w["dv"], w["n_slots"], w["dtype"],
                           w["seed"], device, w.get("pool_std", 0.02), decay_scale)
    return make_prefill(w["lens"], w["H"], w["dk"], w["dv"], w["dtype"], w["seed"], device,
                        w.get("init_std"), decay_scale, beta_scale)
