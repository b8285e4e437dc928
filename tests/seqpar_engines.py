"""The fp64 oracle as a segment engine for the sequence-parallel host logic
(test infrastructure: only tests use it)."""
import torch

import oracle
from sliding_window_softmax_gb300.seqpar import Engine


def _t(a):
    return torch.from_numpy(a)


def oracle_engine() -> Engine:
    def fwd(q, k, v, la, w, h0):
        o, lse, hk, hv = oracle.forward(q, k, v, la, w, h0=h0, return_state=True)
        return _t(o), _t(lse), (_t(hk), _t(hv))

    def bwd(q, k, v, la, o, lse, dout, w, h0, dhT):
        g = oracle.backward(q, k, v, la, dout, w, h0=h0, dhT=dhT)
        return tuple(_t(x) for x in g[:4]) + (((_t(g[4]), _t(g[5])) if h0 is not None else None),)

    def decay(la, w):
        T = la.shape[2]
        return torch.exp(la[:, :, :max(T - w, 0)].double().sum(2))

    def combine(a, prev, cur):
        return tuple(a[..., None] * p + c for p, c in zip(prev, cur))

    return Engine(fwd, bwd, decay, combine)
