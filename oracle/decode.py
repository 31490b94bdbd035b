"""TEST INFRASTRUCTURE ONLY: the SFI decode loop run on the CPU oracle.

Follows the pages' step order ("How SFI Works" in the blog; sections 2A-2C and 3 of the
gist.science technical summary): every step appends the new token; a slow step runs
dense attention, turns its weights into the Selector's evidence, fuses it with the
positional prior and keeps the Top-K; a fast step attends to sinks + selected memory +
the sliding recent window. The step type comes from the trigger policy on the boundary
mask. Units (layer, sequence, kv head) are independent, so a subset can be simulated.
"""
from __future__ import annotations

import time

import numpy as np

import oracle


def epochs(mask: np.ndarray) -> np.ndarray:
    """epoch[t] = number of boundary tokens before step t (drifting heavy hitters)."""
    e = np.zeros(mask.shape[0], dtype=np.int64)
    e[1:] = np.cumsum(mask[:-1])
    return e


def schedule(wl, steps: int | None = None) -> np.ndarray:
    """Slow flags [B][steps] by the oracle's trigger policy: on the workload's boundary masks,
    or, for a token-triggered workload, on its generated token streams (trigger tokens
    '.', '?', '!', newline; gist.science summary, section 2C)."""
    cfg = wl.cfg
    n = cfg.steps if steps is None else steps
    if cfg.trigger == "tokens":
        from synth.gen import TRIGGER_TOKENS
        trig = np.asarray(TRIGGER_TOKENS, np.int32)
        return np.stack([oracle.schedule_tokens(wl.tokens[b][:n], trig, cfg.t_max)
                         for b in range(cfg.batch)])
    return np.stack([oracle.schedule(wl.masks[b][:n], cfg.t_max) for b in range(cfg.batch)])


def _sub(kc, vc, idx):
    """The caches of the units in idx (no copy when that is every unit)."""
    if len(idx) == kc.shape[0]:
        return kc, vc
    return kc[idx], vc[idx]


def prepare(wl, steps: int, units=None):
    """Generate (untimed) the K/V rows every simulated unit will read: prefill + appended."""
    cfg = wl.cfg
    units = list(range(wl.n_units)) if units is None else list(units)
    coords = []
    for u in units:
        kvh = u % cfg.n_kv_heads
        b = (u // cfg.n_kv_heads) % cfg.batch
        layer = u // (cfg.n_kv_heads * cfg.batch)
        coords.append((layer, b, kvh))
    cap = int(max(wl.len0)) + steps
    kc = np.zeros((len(units), cap, cfg.head_dim), np.uint16)
    vc = np.zeros((len(units), cap, cfg.head_dim), np.uint16)
    for i, (layer, b, kvh) in enumerate(coords):
        n = int(wl.len0[b]) + steps
        kc[i, :n] = wl.rows("k", layer, b, kvh, np.arange(n))
        vc[i, :n] = wl.rows("v", layer, b, kvh, np.arange(n))
    return {"units": units, "coords": coords, "k": kc, "v": vc, "steps": steps}


def run(wl, steps: int | None = None, units=None, threads: int = 0, want_f: bool = False,
        gpu_selection=None, prepared=None, slow=None):
    """Simulate `steps` decode steps for the given units (default: all).

    slow (optional): uint8 [B][steps] step types to use instead of the trigger policy's
    (a benchmark sample of one slow step and the fast steps that follow it).

    gpu_selection (optional): {(t, u): ascending positions} to use instead of the oracle's
    own selection at slow steps (isolates the attention from selection near-ties).
    Returns dict with 'slow' [B][steps], 'out' {t: [n_units][G][D] double},
    'sel' {(t, u): positions}, 'f' {(t, u): fp32 evidence} when want_f."""
    cfg = wl.cfg
    steps = cfg.steps if steps is None else steps
    if prepared is None or prepared["steps"] < steps:
        prepared = prepare(wl, steps, units)
    units, coords = prepared["units"], prepared["coords"]
    kc, vc = prepared["k"], prepared["v"]
    G, D = cfg.group, cfg.head_dim
    S, W, K = cfg.n_sink, cfg.n_window, cfg.n_select
    nU = len(units)
    slow = schedule(wl, steps) if slow is None else np.asarray(slow, np.uint8)[:, :steps]
    ep = np.stack([epochs(wl.masks[b][:steps]) for b in range(cfg.batch)])
    L_slow = np.zeros(nU, np.int64)
    sel = [np.zeros(0, np.int32) for _ in range(nU)]
    res = {"slow": slow, "out": {}, "sel": {}, "f": {}, "seconds": np.zeros(steps)}
    qcache = {}
    for t in range(steps):
        # input generation and the drifting-key edits are harness work: not timed
        if cfg.drift and t > 0:
            for i, (layer, b, kvh) in enumerate(coords):
                if ep[b, t] != ep[b, t - 1]:
                    old = wl.hh_positions(layer, b, kvh, int(ep[b, t - 1]))
                    new = wl.hh_positions(layer, b, kvh, int(ep[b, t]))
                    ch = np.union1d(old, new)
                    kc[i, ch] = wl.rows("k", layer, b, kvh, ch, epoch=int(ep[b, t]))
        for (layer, b) in {(layer, b) for (layer, b, _) in coords}:
            qcache[(layer, b)] = wl.query(t, layer, b)
        q = np.stack([qcache[(layer, b)][kvh * G:(kvh + 1) * G] for (layer, b, kvh) in coords])
        L = np.array([int(wl.len0[b]) + t + 1 for (_, b, _) in coords], np.int64)
        is_slow = np.array([slow[b, t] for (_, b, _) in coords], bool)
        t0 = time.perf_counter()
        out = np.zeros((nU, G, D))
        if is_slow.any():
            idx = np.flatnonzero(is_slow)
            o, f = oracle.attend_batch(q[idx], *_sub(kc, vc, idx), L[idx], want_f=True,
                                       threads=threads)
            out[idx] = o
            for j, i in enumerate(idx):
                f32 = f[j, :L[i]].astype(np.float32)
                if gpu_selection is not None and (t, units[i]) in gpu_selection:
                    sel[i] = np.asarray(gpu_selection[(t, units[i])], np.int32)
                else:
                    sel[i] = oracle.select(int(L[i]), S, W, K, cfg.prior_tau, cfg.lam, f32)
                L_slow[i] = L[i]
                res["sel"][(t, units[i])] = sel[i]
                if want_f:
                    res["f"][(t, units[i])] = f32
        if (~is_slow).any():
            idx = np.flatnonzero(~is_slow)
            rows = [oracle.sparse_rows(int(L_slow[i]), int(L[i]), S, W, sel[i]) for i in idx]
            rmax = max(len(r) for r in rows)
            rr = np.zeros((len(idx), rmax), np.int32)
            for j, r in enumerate(rows):
                rr[j, :len(r)] = r
            o, _ = oracle.attend_batch(q[idx], *_sub(kc, vc, idx),
                                       np.array([len(r) for r in rows]), rows=rr,
                                       threads=threads)
            out[idx] = o
        res["out"][t] = out
        res["seconds"][t] = time.perf_counter() - t0
    return res
