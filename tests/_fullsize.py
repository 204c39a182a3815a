"""Helpers of the full-size parity tests: host copies of one expert's bf16 weights, a process
pool for the oracle's per-expert work, and a token sample that reaches every active expert.

The oracle's MXFP8 weight quantiser takes about a second per full-size weight in numpy, so the
full-size checks run the oracle's per-expert work (its ``expert_map`` argument) in a pool of
processes started with ``spawn`` (never forked after CUDA has been initialised).  Each job
carries one expert's weights as raw bf16 bits (2 bytes per element), converted to float64
exactly inside the worker."""

import contextlib
import os

import numpy as np


class BF16Bits:
    """Raw bfloat16 bits (uint16) of one weight matrix; np.asarray(..., float64) gives its exact
    values (a bf16 value is the upper half of the float32 with the same bits)."""

    def __init__(self, bits):
        self.bits = bits

    def __array__(self, dtype=None, copy=None):
        a = (self.bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        return a if dtype is None else a.astype(dtype, copy=False)


class HostExperts:
    """Indexable view of a stacked [E, a, b] bf16 CUDA tensor: expert e's bits copied to the
    host on access."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        import torch

        bits = self.t[e].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return BF16Bits(bits)


@contextlib.contextmanager
def oracle_pool(processes=None):
    """``expert_map`` for the oracle: an ordered imap over a spawn-started process pool."""
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    with ctx.Pool(processes or os.cpu_count()) as pool:
        yield lambda fn, jobs: pool.imap(fn, jobs, chunksize=1)


def cover_tokens(idx, n_min, must=()):
    """Sorted token ids: the tokens of `must`, then tokens chosen greedily (most experts not yet
    reached first) until every expert that any token selects is selected by a chosen token,
    then evenly spaced tokens up to n_min in all."""
    idx = np.asarray(idx)
    T = idx.shape[0]
    chosen = list(dict.fromkeys(int(t) for t in must))
    need = set(idx.ravel().tolist()) - set(idx[chosen].ravel().tolist())
    while need:
        gain = np.isin(idx, list(need)).sum(axis=1)
        gain[chosen] = -1
        t = int(np.argmax(gain))
        chosen.append(t)
        need -= set(idx[t].tolist())
    for t in np.linspace(0, T - 1, num=min(T, n_min) + 2).astype(int)[1:-1]:
        if len(chosen) >= n_min:
            break
        if int(t) not in chosen:
            chosen.append(int(t))
    return sorted(chosen)


def most_experts_tokens(idx, n):
    """n token ids chosen greedily to reach as many distinct experts as possible."""
    idx = np.asarray(idx)
    chosen, seen = [], set()
    for _ in range(min(n, idx.shape[0])):
        gain = np.array([len(set(r.tolist()) - seen) for r in idx])
        gain[chosen] = -1
        t = int(np.argmax(gain))
        chosen.append(t)
        seen |= set(idx[t].tolist())
    return sorted(chosen)


def experts_of(L):
    return HostExperts(L["W_gate"]), HostExperts(L["W_up"]), HostExperts(L["W_down"])


def sampled_tokens(got, counts, T):
    """At least 64 tokens reaching every active expert, the hottest expert's first token first."""
    hot = int(np.argmax(counts))
    toks = cover_tokens(got, 64, must=[0, T - 1, int(np.nonzero((got == hot).any(1))[0][0])])
    assert set(got[toks].ravel().tolist()) == set(np.nonzero(counts)[0].tolist())
    return toks


def dw_experts(counts):
    """Hottest, least busy non-empty, median non-empty, and one whose rows end mid-tile."""
    nz = np.nonzero(counts)[0]
    by = nz[np.argsort(counts[nz], kind="stable")]
    picks = [int(by[-1]), int(by[0]), int(by[len(by) // 2])]
    mid = [int(e) for e in by if 0 < counts[e] % 128 < 64 and counts[e] > 128 and int(e) not in picks]
    if mid:
        picks.append(mid[0])
    return picks
