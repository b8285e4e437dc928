"""One sequence cut into segments: sequence parallelism for the NHA operator.

A sequence of T tokens is cut into segments [a_r, b_r).  Segment r runs the
operator on its *extended* range [lo_r, b_r), lo_r = max(0, a_r - w): the w
tokens before it (its halo) and its own tokens.  Its queries in the halo
are dropped; its own queries then see exactly their full-sequence window,
and its long memory must start from h0_r = the long memory after token
lo_r - 1 (the Paper-Notes page's chunkwise form carries the long memory from
chunk to chunk; here it is carried from segment to segment).

The long memory is a linear recurrence, so h0 follows from per-segment
summaries by an associative scan: with S_r the final state of segment r's run
started from zero states and A_r the product of the gates of its tokens that
left the window (per slot),

    h0_{r+1} = A_r o h0_r + S_r.

Every segment forms its summary independently; the scan over the summaries
and the halo are the only exchange.  In the backward the state adjoint runs
the other way, g_r = dh0_r + A_r o g_{r+1}, and segment r's gradient with
respect to its final state is g_{r+1}; the halo tokens' gradients go back to
the segment that owns them.

The arithmetic runs in an *engine* (the library's CUDA kernels by default:
nha_forward / nha_backward with slot states, nha_gate_total,
nha_state_combine); this module only slices, orders and exchanges.
:func:`forward_segments` / :func:`backward_segments` run every segment in one
process; :func:`forward_rank` / :func:`backward_rank` run one segment per rank
of a torch.distributed process group, with all_gather as the exchange.
(The Paper-Notes page, 局限, names contexts beyond 128K as unvalidated: this is
the split such contexts need across devices.)
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional, Sequence, Tuple

import torch

State = Tuple[torch.Tensor, torch.Tensor]  # (K part, V part), fp32 [B, H, m, d]


@dataclasses.dataclass(frozen=True)
class Segment:
    lo: int  # first token of the extended run (halo start)
    a: int   # first own token
    b: int   # one past the last own token

    @property
    def keep(self) -> int:
        """Rows of the extended run before the own tokens (the halo)."""
        return self.a - self.lo


def segment_plan(T: int, n: int, w: int) -> List[Segment]:
    """n contiguous segments of T tokens (sizes differing by at most one)."""
    if n <= 0 or T < n:
        raise ValueError(f"cannot cut {T} tokens into {n} segments")
    base, extra = divmod(T, n)
    out, a = [], 0
    for r in range(n):
        b = a + base + (1 if r < extra else 0)
        out.append(Segment(max(0, a - max(int(w), 0)), a, b))
        a = b
    return out


@dataclasses.dataclass
class Engine:
    """The arithmetic of one segment, on tensors [B, H, T, *]."""
    # (q, k, v, log_alpha, w, h0) -> (o, lse, hT)
    forward: Callable
    # (q, k, v, log_alpha, o, lse, dout, w, h0, dhT) -> (dq, dk, dv, dlog_alpha, dh0 or None)
    backward: Callable
    # (log_alpha, w) -> decay [B, H, m]
    decay: Callable
    # (decay, prev, cur) -> decay o prev + cur
    combine: Callable


def library_engine() -> Engine:
    """The library's kernels (CUDA tensors)."""
    from . import _binding as nb

    def fwd(q, k, v, la, w, h0):
        return nb.nha_forward(q, k, v, la, w=w, h0=h0, return_state=True)

    def bwd(q, k, v, la, o, lse, dout, w, h0, dhT):
        g = nb.nha_backward(q, k, v, la, o, lse, dout, w=w, h0=h0, dhT=dhT)
        return tuple(g[:4]) + ((g[4], g[5]) if h0 is not None else None,)

    return Engine(fwd, bwd, lambda la, w: nb.nha_gate_total(la, w),
                  lambda a, prev, cur: nb.nha_state_combine(a, prev, cur))


def initial_states(summaries: Sequence[Tuple[torch.Tensor, State]], starts: Sequence[int],
                   combine) -> List[Optional[State]]:
    """Exclusive scan: h0 of every segment from the (A_r, S_r) of the ones
    before it.  A run that starts at token 0 (starts[r] == 0: the first, or one
    whose halo reaches back to the start) has no long memory before it (None)
    and re-forms everything before it itself."""
    h0: List[Optional[State]] = []
    for r, lo in enumerate(starts):
        if lo == 0:
            h0.append(None)
        else:
            A, S = summaries[r - 1]
            prev = h0[r - 1]
            h0.append(S if prev is None else combine(A, prev, S))
    return h0


def final_state_gradients(dh0: Sequence[Optional[State]], decays: Sequence[torch.Tensor],
                          starts: Sequence[int], combine) -> List[Optional[State]]:
    """Reverse scan: the gradient with respect to segment r's final state, g_{r+1}
    with g_r = dh0_r + A_r o g_{r+1}, where segment r + 1 starts from segment r's
    final state (None otherwise: for the last segment, and before a run that
    starts at token 0)."""
    n = len(dh0)
    dhT: List[Optional[State]] = [None] * n
    g = None  # the gradient with respect to h0 of the segment after r
    for r in range(n - 1, -1, -1):
        if r + 1 < n and starts[r + 1] > 0:
            dhT[r] = g
        if starts[r] == 0:
            g = None  # segment r has no h0: nothing flows further back
        else:
            g = dh0[r] if dhT[r] is None else combine(decays[r], dhT[r], dh0[r])
    return dhT


def _ext(x: dict, s: Segment) -> dict:
    return {n: t[:, :, s.lo:s.b].contiguous() for n, t in x.items()}


def forward_segments(q, k, v, log_alpha, w: int, n: int, engine: Optional[Engine] = None):
    """o, lse of the whole sequence, computed segment by segment; returns
    (o, lse, ctx) with ctx for :func:`backward_segments`."""
    eng = engine or library_engine()
    plan = segment_plan(q.shape[2], n, w)
    x = dict(q=q, k=k, v=v, la=log_alpha)
    ext = [_ext(x, s) for s in plan]
    # summaries: each run from zero states (its h0 does not matter for them)
    summ = []
    for e in ext[:-1]:
        _, _, S = eng.forward(e["q"], e["k"], e["v"], e["la"], w, None)
        summ.append((eng.decay(e["la"], w), S))
    summ.append((None, None))
    starts = [s.lo for s in plan]
    h0 = initial_states(summ, starts, eng.combine)
    o = lse = None
    runs = []
    for s, e, h in zip(plan, ext, h0):
        oe, le, _ = eng.forward(e["q"], e["k"], e["v"], e["la"], w, h)
        if o is None:
            o = torch.empty(q.shape, dtype=oe.dtype, device=oe.device)
            lse = torch.empty(q.shape[:3], dtype=le.dtype, device=le.device)
        o[:, :, s.a:s.b] = oe[:, :, s.keep:]
        lse[:, :, s.a:s.b] = le[:, :, s.keep:]
        runs.append((oe, le))
    decays = [A for A, _ in summ]
    return o, lse, dict(plan=plan, ext=ext, h0=h0, runs=runs, decays=decays, w=w, starts=starts)


def backward_segments(ctx: dict, dout, engine: Optional[Engine] = None):
    """dq, dk, dv, dlog_alpha of <o, dout> for :func:`forward_segments`'s o."""
    eng = engine or library_engine()
    plan, ext, h0, runs, w = ctx["plan"], ctx["ext"], ctx["h0"], ctx["runs"], ctx["w"]
    grads = [None] * len(plan)
    dh0 = [None] * len(plan)
    for r, (s, e, h, (oe, le)) in enumerate(zip(plan, ext, h0, runs)):
        de = torch.zeros_like(oe)
        de[:, :, s.keep:] = dout[:, :, s.a:s.b]
        g = eng.backward(e["q"], e["k"], e["v"], e["la"], oe, le, de, w, h, None)
        grads[r], dh0[r] = list(g[:4]), g[4]
    dhT = final_state_gradients(dh0, ctx["decays"], ctx["starts"], eng.combine)
    for r, (s, e, h, (oe, le)) in enumerate(zip(plan, ext, h0, runs)):
        if dhT[r] is None:
            continue
        g = eng.backward(e["q"], e["k"], e["v"], e["la"], oe, le, torch.zeros_like(oe), w, h, dhT[r])
        for i in range(4):
            grads[r][i] = grads[r][i] + g[i]
    q = ctx["ext"][0]["q"]
    B, H = q.shape[:2]
    T = plan[-1].b
    out = [torch.zeros((B, H, T) + t.shape[3:], dtype=t.dtype, device=t.device) for t in grads[0]]
    for s, g in zip(plan, grads):
        for i in range(4):
            out[i][:, :, s.lo:s.b] += g[i]  # the halo rows add into the segment that owns them
    return tuple(out)


# ------------------------------------------------------------------------------------------
# One segment per rank of a process group (torch.distributed; all_gather exchanges).
def _gather(t: torch.Tensor) -> List[torch.Tensor]:
    import torch.distributed as dist

    out = [torch.empty_like(t) for _ in range(dist.get_world_size())]
    dist.all_gather(out, t.contiguous())
    return out


def _halo(x: torch.Tensor, w: int, rank: int) -> torch.Tensor:
    """The w rows (dim 2) just before this rank's tokens: the last w of the
    previous rank's (every rank holds at least w tokens)."""
    tails = _gather(x[:, :, x.shape[2] - w:])
    return tails[rank - 1] if rank > 0 else x[:, :, :0]


def forward_rank(q, k, v, log_alpha, w: int, engine: Optional[Engine] = None):
    """This rank's o, lse for its own tokens (rank r holds the r-th of consecutive
    segments, each at least w tokens long); returns (o, lse, ctx)."""
    import torch.distributed as dist

    eng = engine or library_engine()
    rank, world = dist.get_rank(), dist.get_world_size()
    sizes = _gather(torch.tensor([q.shape[2]], device=q.device))
    if min(int(n) for n in sizes) < w:
        raise ValueError(f"every rank must hold at least w = {w} tokens, got {[int(n) for n in sizes]}")
    halo = {n: _halo(t, w, rank) for n, t in dict(q=q, k=k, v=v, la=log_alpha).items()}
    e = {n: torch.cat([halo[n], t], dim=2) for n, t in dict(q=q, k=k, v=v, la=log_alpha).items()}
    keep = halo["q"].shape[2]
    _, _, S = eng.forward(e["q"], e["k"], e["v"], e["la"], w, None)
    A = eng.decay(e["la"], w)
    As, Sk, Sv = _gather(A), _gather(S[0]), _gather(S[1])
    summ = [(As[r], (Sk[r], Sv[r])) for r in range(world)]
    # run r starts at token (sum of the sizes before it) - w
    starts, a = [], 0
    for r in range(world):
        starts.append(max(0, a - w))
        a += int(sizes[r])
    h0 = initial_states(summ, starts, eng.combine)[rank]
    oe, le, _ = eng.forward(e["q"], e["k"], e["v"], e["la"], w, h0)
    ctx = dict(ext=e, keep=keep, h0=h0, o=oe, lse=le, decays=As, w=w, starts=starts, state_like=S[0])
    return oe[:, :, keep:], le[:, :, keep:], ctx


def backward_rank(ctx: dict, dout, engine: Optional[Engine] = None):
    """This rank's dq, dk, dv, dlog_alpha for its own tokens."""
    import torch.distributed as dist

    eng = engine or library_engine()
    rank, world = dist.get_rank(), dist.get_world_size()
    e, keep, h0, oe, le, w = ctx["ext"], ctx["keep"], ctx["h0"], ctx["o"], ctx["lse"], ctx["w"]
    de = torch.zeros_like(oe)
    de[:, :, keep:] = dout
    g = eng.backward(e["q"], e["k"], e["v"], e["la"], oe, le, de, w, h0, None)
    grads, dh0 = list(g[:4]), g[4]
    zero = torch.zeros_like(ctx["state_like"])  # the summaries' layout and type
    dk0, dv0 = _gather(dh0[0] if dh0 is not None else zero), _gather(dh0[1] if dh0 is not None else zero)
    starts = ctx["starts"]
    dh0_all = [None if starts[r] == 0 else (dk0[r], dv0[r]) for r in range(world)]
    dhT = final_state_gradients(dh0_all, list(ctx["decays"]), starts, eng.combine)[rank]
    if dhT is not None:
        c = eng.backward(e["q"], e["k"], e["v"], e["la"], oe, le, torch.zeros_like(oe), w, h0, dhT)
        for i in range(4):
            grads[i] = grads[i] + c[i]
    # halo rows go back to the rank that owns them: rank r's halo is the last w
    # tokens of rank r - 1
    out = []
    for t in grads:
        own = t[:, :, keep:].clone()
        halos = _gather(t[:, :, :w] if keep == w else torch.zeros_like(t[:, :, :w]))
        if rank + 1 < world and w > 0:
            own[:, :, own.shape[2] - w:] += halos[rank + 1]
        out.append(own)
    return tuple(out)
