"""Host view of one synthetic workload: prefill lengths, boundary masks, page tables and
on-demand bf16 rows of K, V and queries. Everything is a pure function of the workload's
seed, so any (layer, sequence, head, position) slice can be regenerated without holding
the whole cache."""
from __future__ import annotations

import numpy as np

from . import gen
from .configs import Workload


class HostWorkload:
    def __init__(self, cfg: Workload):
        self.cfg = cfg
        self.key = gen.key_from_seed(cfg.seed)
        B = cfg.batch
        if cfg.ctx_lo == cfg.ctx:
            self.len0 = np.full(B, cfg.ctx, dtype=np.int64)
        else:
            self.len0 = gen.ragged_lengths(self.key, B, cfg.ctx_lo, cfg.ctx)
        self.tokens = None
        if cfg.trigger == "tokens":
            # generated token ids [B][steps]; masks[b][t] = 1 where token t is a trigger
            ts = [gen.token_stream(self.key, cfg.steps, mean_span=cfg.mask_param,
                                   b=b if cfg.per_seq_mask else 0) for b in range(B)]
            self.tokens = np.stack(ts).astype(np.int32)
            self.masks = np.isin(self.tokens, gen.TRIGGER_TOKENS).astype(np.uint8)
        elif cfg.per_seq_mask:
            self.masks = np.stack([gen.boundary_mask(self.key, cfg.steps, cfg.mask_kind,
                                                     cfg.mask_param, b) for b in range(B)])
        else:
            m = gen.boundary_mask(self.key, cfg.steps, cfg.mask_kind, cfg.mask_param, 0)
            self.masks = np.stack([m] * B)
        if cfg.key_model == "hh":
            self.qa, self.ka = gen.hh_direction(self.key, cfg.n_layers, cfg.n_kv_heads,
                                                cfg.head_dim)
        else:
            self.qa = self.ka = None
        self._hh = {}
        if cfg.page_size:
            self.table, self.n_pages = gen.page_table(self.key, self.len0 + cfg.steps,
                                                      cfg.page_size)
        else:
            self.table, self.n_pages = None, 0

    # -- structure ------------------------------------------------------------------------
    @property
    def n_units(self) -> int:
        c = self.cfg
        return c.n_layers * c.batch * c.n_kv_heads

    def unit_index(self, layer: int, b: int, kvh: int) -> int:
        c = self.cfg
        return (layer * c.batch + b) * c.n_kv_heads + kvh

    def n_epochs(self) -> int:
        """Heavy-hitter epochs a run can reach (one more per boundary token)."""
        return 1 + int(self.masks.sum(axis=1).max()) if self.cfg.drift else 1

    def hh_positions(self, layer: int, b: int, kvh: int, epoch: int = 0) -> np.ndarray:
        k = (layer, b, kvh)
        if k not in self._hh or len(self._hh[k]) <= epoch:
            self._hh[k] = gen.hh_epochs(self.key, layer, b, kvh, self.cfg.ctx,
                                        max(epoch + 1, self.n_epochs()))
        return self._hh[k][epoch]

    # -- content --------------------------------------------------------------------------
    def rows(self, which: str, layer: int, b: int, kvh: int, positions, epoch: int = 0):
        """bf16 bits [n][D] of cache rows (prefill or appended tokens alike)."""
        c = self.cfg
        positions = np.asarray(positions, dtype=np.int64)
        if c.key_model == "hh":
            hh = np.isin(positions, self.hh_positions(layer, b, kvh, epoch))
            return gen.kv_rows(self.key, which, layer, b, kvh, positions, c.head_dim, "hh",
                               self.ka[layer, kvh], hh)
        return gen.kv_rows(self.key, which, layer, b, kvh, positions, c.head_dim, c.key_model)

    def query(self, step: int, layer: int, b: int):
        """bf16 bits [Hq][D] of the decode query of `step`."""
        c = self.cfg
        qa = None if self.qa is None else self.qa[layer]
        return gen.q_rows(self.key, step, layer, b, c.n_q_heads, c.head_dim, qa, c.group)

    # -- dense host arrays (small workloads only) ------------------------------------------
    def cache_contiguous(self, which: str, capacity: int | None = None, fill=None):
        """bf16 bits [Ly][B][Hkv][cap][D]; rows below fill[b] (default: prefill length)."""
        c = self.cfg
        cap = capacity or c.capacity
        fill = self.len0 if fill is None else np.asarray(fill)
        out = np.zeros((c.n_layers, c.batch, c.n_kv_heads, cap, c.head_dim), dtype=np.uint16)
        for l in range(c.n_layers):
            for b in range(c.batch):
                for h in range(c.n_kv_heads):
                    out[l, b, h, :fill[b]] = self.rows(which, l, b, h, np.arange(fill[b]))
        return out

    def cache_paged(self, which: str, fill=None):
        """bf16 bits [Ly][n_pages][Hkv][page][D] laid out through the page table."""
        c = self.cfg
        ps = c.page_size
        fill = self.len0 if fill is None else np.asarray(fill)
        out = np.zeros((c.n_layers, self.n_pages, c.n_kv_heads, ps, c.head_dim), dtype=np.uint16)
        for l in range(c.n_layers):
            for b in range(c.batch):
                pos = np.arange(fill[b])
                pages = self.table[b, pos // ps]
                for h in range(c.n_kv_heads):
                    out[l, pages, h, pos % ps] = self.rows(which, l, b, h, pos)
        return out

    def queries(self, steps: int | None = None):
        """bf16 bits [steps][Ly][B][Hq][D]."""
        c = self.cfg
        n = c.steps if steps is None else steps
        out = np.zeros((n, c.n_layers, c.batch, c.n_q_heads, c.head_dim), dtype=np.uint16)
        for t in range(n):
            for l in range(c.n_layers):
                for b in range(c.batch):
                    out[t, l, b] = self.query(t, l, b)
        return out

    def new_tokens(self, which: str, steps: int | None = None):
        """bf16 bits [steps][Ly][B][Hkv][D]: the row appended at step t is position len0[b]+t."""
        c = self.cfg
        n = c.steps if steps is None else steps
        out = np.zeros((n, c.n_layers, c.batch, c.n_kv_heads, c.head_dim), dtype=np.uint16)
        for l in range(c.n_layers):
            for b in range(c.batch):
                pos = self.len0[b] + np.arange(n)
                for h in range(c.n_kv_heads):
                    out[:, l, b, h] = self.rows(which, l, b, h, pos)
        return out
