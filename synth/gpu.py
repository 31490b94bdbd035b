"""Device-side filling of workload tensors through synth/libsynth.so (the GPU twin of
synth.gen). Used by the benchmark and the GPU tests to build large caches in place."""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import gen

_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsynth.so")
_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB):
            raise RuntimeError(f"{_LIB} is missing: build it with __graft_entry__.build()")
        l = C.CDLL(_LIB)
        P, I, U64 = C.c_void_p, C.c_int, C.c_uint64
        l.synth_fill_contig.argtypes = [P, I, I, I, I, I, P, U64, I, P, P, I, P, P, I, P]
        l.synth_fill_paged.argtypes = [P, I, I, I, I, I, P, P, P, U64, I, P, P, I, P, P, I, P]
        l.synth_fill_new.argtypes = [P, I, I, I, I, I, P, U64, I, P, P, I, P, P, I, P]
        l.synth_fill_queries.argtypes = [P, I, I, I, I, I, U64, P, P]
        _lib = l
    return _lib


class DeviceModel:
    """Device copies of the key-model tables of a HostWorkload."""

    def __init__(self, wl, device, epoch_positions=None):
        import torch
        cfg = wl.cfg
        self.kind = {"zipf": 1, "hh": 2}.get(cfg.key_model, 0)
        thr, boosts = gen.zipf_tables()
        self.zthr = torch.from_numpy(thr.view(np.int32).copy()).to(device)
        self.zboost = torch.from_numpy(boosts).to(device)
        self.zkmax = int(thr.shape[0])
        self.ka = self.qa = self.bits = None
        self.words = 1
        if self.kind == 2:
            self.ka = torch.from_numpy(wl.ka.copy()).to(device)
            self.qa = torch.from_numpy(wl.qa.copy()).to(device)
            cap = int(max(wl.len0)) + cfg.steps
            pos = []
            for layer in range(cfg.n_layers):
                for b in range(cfg.batch):
                    for h in range(cfg.n_kv_heads):
                        ep = 0 if epoch_positions is None else epoch_positions(layer, b, h)
                        pos.append(wl.hh_positions(layer, b, h, ep))
            bm = gen.hh_bitmap(pos, cap)
            self.words = bm.shape[1]
            self.bits = torch.from_numpy(bm.view(np.int32)).to(device)

    def args(self):
        p = lambda t: None if t is None else t.data_ptr()
        return (self.kind, p(self.zthr), p(self.zboost), self.zkmax, p(self.ka), p(self.bits),
                self.words)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed with CUDA error {rc}")


def fill_cache(wl, k, v, fill_len, model: DeviceModel, page_owner=None, stream=0):
    """Fill the device cache tensors k, v (contiguous or paged) with the workload's rows for
    positions below fill_len[b] (device int64 [B]); other rows are zeroed."""
    cfg = wl.cfg
    key = int(wl.key)
    for stream_id, t in ((gen.STREAM_K, k), (gen.STREAM_V, v)):
        if cfg.page_size:
            ob, olp = page_owner
            _check(lib().synth_fill_paged(t.data_ptr(), stream_id, cfg.n_layers, cfg.batch,
                                          wl.n_pages, cfg.n_kv_heads, ob.data_ptr(), olp.data_ptr(),
                                          fill_len.data_ptr(), key, *model.args(), stream),
                   "synth_fill_paged")
        else:
            _check(lib().synth_fill_contig(t.data_ptr(), stream_id, cfg.n_layers, cfg.batch,
                                           cfg.n_kv_heads, t.shape[3], fill_len.data_ptr(), key,
                                           *model.args(), stream), "synth_fill_contig")


def fill_new_tokens(wl, k_new, v_new, len0, model: DeviceModel, stream=0):
    cfg = wl.cfg
    for stream_id, t in ((gen.STREAM_K, k_new), (gen.STREAM_V, v_new)):
        _check(lib().synth_fill_new(t.data_ptr(), stream_id, t.shape[0], cfg.n_layers, cfg.batch,
                                    cfg.n_kv_heads, len0.data_ptr(), int(wl.key), *model.args(),
                                    stream), "synth_fill_new")


def fill_queries(wl, q, model: DeviceModel, stream=0):
    cfg = wl.cfg
    qa = None if model.qa is None else model.qa.data_ptr()
    _check(lib().synth_fill_queries(q.data_ptr(), q.shape[0], cfg.n_layers, cfg.batch,
                                    cfg.n_q_heads, cfg.group, int(wl.key), qa, stream),
           "synth_fill_queries")


def page_owners(wl, device):
    """Reverse page table: owner sequence and logical page of every physical page."""
    import torch
    ob = np.full(wl.n_pages, -1, np.int32)
    olp = np.zeros(wl.n_pages, np.int32)
    for b in range(wl.cfg.batch):
        for lp, pg in enumerate(wl.table[b]):
            if pg >= 0:
                ob[pg] = b
                olp[pg] = lp
    return torch.from_numpy(ob).to(device), torch.from_numpy(olp).to(device)


def drift_edits(wl, device):
    """Per boundary epoch e >= 1: device arrays (pos [U][m], planted [U][m]) listing the
    K rows whose heavy-hitter membership changes from epoch e-1 to e."""
    import torch
    cfg = wl.cfg
    U = wl.n_units
    n_ep = wl.n_epochs()
    per_unit = []
    for layer in range(cfg.n_layers):
        for b in range(cfg.batch):
            for h in range(cfg.n_kv_heads):
                per_unit.append([wl.hh_positions(layer, b, h, e) for e in range(n_ep)])
    out = {}
    # epoch e >= 1: changes from e-1 to e; key 0: back from the last epoch to epoch 0
    for e in range(0, n_ep):
        if e == 0 and n_ep == 1:
            continue
        changes = []
        for u in range(U):
            old = per_unit[u][e - 1] if e > 0 else per_unit[u][n_ep - 1]
            new = per_unit[u][e]
            ch = np.setxor1d(old, new)
            changes.append((ch, np.isin(ch, new)))
        m = max(1, max(len(c[0]) for c in changes))
        pos = np.full((U, m), -1, np.int32)
        pl = np.zeros((U, m), np.uint8)
        for u, (ch, f) in enumerate(changes):
            pos[u, :len(ch)] = ch
            pl[u, :len(ch)] = f
        out[e] = (torch.from_numpy(pos).to(device), torch.from_numpy(pl).to(device), m)
    return out


def apply_drift(wl, k, edit, model: "DeviceModel", stream=0):
    """Rewrite the changed K rows of one epoch (edit from drift_edits)."""
    cfg = wl.cfg
    pos, pl, m = edit
    l = lib()
    if not hasattr(l, "_rewrite_set"):
        l.synth_rewrite_k.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p, C.c_int,
                                      C.c_int, C.c_int, C.c_uint64, C.c_void_p, C.c_void_p]
        l._rewrite_set = True
    _check(l.synth_rewrite_k(k.data_ptr(), wl.n_units, m, pos.data_ptr(), pl.data_ptr(), cfg.batch,
                             cfg.n_kv_heads, k.shape[3], int(wl.key), model.ka.data_ptr(), stream),
           "synth_rewrite_k")
