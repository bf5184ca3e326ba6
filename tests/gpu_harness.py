"""Runs a workload through the C ABI (CUDA path) and, beside it, through the
oracle, step by step, and compares them.  Inputs for both sides come from
the seeded generators in ``workloads`` (generated on the GPU, copied to the
host for the oracle); no expected value comes from the CUDA path."""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle as O
import paged_kv_cache_flash_gb300 as K
import workloads as W

OUT_TOL = 2e-2      # attention output, max abs (bf16 in, fp32 accumulate)
MASS_TOL = 1e-4     # block mass, abs
SCORE_TOL = 1e-5    # EMA score and priority, abs
CUT_MARGIN = 1e-5   # blocks with oracle P this close to a cut are excluded
TOUCH_MARGIN = 1e-5 # blocks with oracle M*nb this close to 1 are excluded


def seq_ids_for(wl):
    # descending ids: call order differs from the ascending-id record order
    return [5000 - 17 * s for s in range(wl.nseq)]


@dataclass
class OracleSeq:
    seq_id: int
    Kbuf: torch.Tensor            # host bf16 [capacity][L][Hkv][d]
    Vbuf: torch.Tensor
    n: int                        # tokens so far
    rec: np.ndarray               # oracle records, block order
    ambiguous: np.ndarray         # touch decision within TOUCH_MARGIN at some step
    page_of: list = field(default_factory=list)   # page identity per block

    @property
    def K(self):
        return self.Kbuf[: self.n]

    @property
    def V(self):
        return self.Vbuf[: self.n]


class Run:
    """oracle_seqs: indices of the sequences the oracle follows (None = all);
    each sequence's attention, mass and records depend on it alone."""

    def __init__(self, wl, alpha, *, staging_pages=8, chunk=4096, oracle_on=True,
                 oracle_seqs=None, pool_pages=None, extra_steps=0, device="cuda",
                 kv_dtype=K.KVS_KV_BF16, k_scale=1.0, v_scale=1.0, kivi_groups=0):
        self.wl, self.alpha = wl, alpha
        self.dev = device
        self.ids = seq_ids_for(wl)
        self.mb = wl.max_blocks_per_seq() + (extra_steps + 15) // 16
        self.fp8 = kv_dtype == K.KVS_KV_FP8_E4M3
        self.kivi = kv_dtype == K.KVS_KV_KIVI2
        self.k_scale, self.v_scale = k_scale, v_scale
        cfg = K.make_config(wl.L, wl.Hq, wl.Hkv, wl.d, pool_pages or wl.pool_pages, max_seqs=wl.nseq,
                            max_blocks_per_seq=self.mb, alpha=alpha,
                            recency_window=wl.recency_window, weights=wl.weights, cuts=wl.cuts,
                            pool_seed=wl.seed, staging_pages=staging_pages, kv_dtype=kv_dtype,
                            k_scale=k_scale, v_scale=v_scale, kivi_groups=kivi_groups)
        self.ctx = K.Context(cfg)
        self.oracle_on = oracle_on
        track = set(range(wl.nseq)) if oracle_seqs is None else set(oracle_seqs)
        self.tracked = [sid for s, sid in enumerate(self.ids) if oracle_on and s in track]
        self.t = 0
        self.ntok = list(wl.prefill_lens)
        self.orc = {}
        B = wl.block_tokens
        pre_blocks = wl.shared_prefix_tokens // B
        cap_steps = wl.steps + extra_steps + 1
        for s, sid in enumerate(self.ids):
            n = wl.prefill_lens[s]
            if s > 0 and pre_blocks:
                self.ctx.seq_add(sid, self.ids[0], pre_blocks)
                start = wl.shared_prefix_tokens
            else:
                self.ctx.seq_add(sid)
                start = 0
            o = None
            if sid in self.tracked:
                shape = (n + cap_steps, wl.L, wl.Hkv, wl.d)
                nb = (n + B - 1) // B
                page_of = [((0, b) if b < pre_blocks else (s, b)) for b in range(nb)]
                o = OracleSeq(sid, torch.empty(shape, dtype=torch.bfloat16),
                              torch.empty(shape, dtype=torch.bfloat16), n,
                              O.new_records(sid, 0, nb, 0), np.zeros(nb, bool), page_of)
                self.orc[sid] = o
            for a in range(0, n, chunk):
                b = min(n, a + chunk)
                if b <= start and o is None:
                    continue
                Kt, Vt = W.kv_tokens(wl, s, a, b, device)
                if o is not None:
                    o.Kbuf[a:b].copy_(Kt.cpu())
                    o.Vbuf[a:b].copy_(Vt.cpu())
                if b > start:
                    lo = max(a, start) - a
                    self.ctx.append_tokens(sid, Kt[lo:].contiguous(), Vt[lo:].contiguous())
                del Kt, Vt
        torch.cuda.synchronize()

    # ------------------------------------------------------------------
    def step(self, gather_host=None, mode=K.KVS_SELECT_THRESH, flags=0, frac=0.0,
             batched_append=True):
        """One decode step over every sequence; returns a dict of GPU results
        and, if the oracle is on, the oracle's.  batched_append: the new
        tokens go in through kvs_append_step (one call), else through one
        kvs_append_tokens call per sequence."""
        wl = self.wl
        B = wl.block_tokens
        self.t += 1
        t = self.t
        new = [W.kv_tokens(wl, s, self.ntok[s], self.ntok[s] + 1, self.dev) for s in range(wl.nseq)]
        if batched_append:
            self.ctx.append_step(self.ids, torch.cat([k for k, _ in new]).contiguous(),
                                 torch.cat([v for _, v in new]).contiguous())
        for s, sid in enumerate(self.ids):
            n = self.ntok[s]
            Kt, Vt = new[s]
            if not batched_append:
                self.ctx.append_tokens(sid, Kt, Vt)
            if sid in self.orc:
                o = self.orc[sid]
                if n % B == 0:      # a new block opens at the step counter t-1
                    o.rec = np.concatenate([o.rec, O.new_records(sid, n // B, 1, t - 1)])
                    o.ambiguous = np.append(o.ambiguous, False)
                    o.page_of.append((s, n // B))
                o.Kbuf[n:n + 1].copy_(Kt.cpu())
                o.Vbuf[n:n + 1].copy_(Vt.cpu())
                o.n = n + 1
            self.ntok[s] = n + 1
        q = torch.stack([W.queries(wl, s, t, self.dev) for s in range(wl.nseq)]).contiguous()
        out = torch.empty((wl.nseq, wl.L, wl.Hq, wl.d), dtype=torch.float32, device=self.dev)
        self.ctx.decode_step(self.ids, q, out)
        self.ctx.score_update()
        res = {"out": out, "q": q}
        nrec = sum((n + B - 1) // B for n in self.ntok)
        ids = torch.zeros(nrec * 2, dtype=torch.int64, device=self.dev)
        slots = torch.full((nrec,), -2, dtype=torch.int32, device=self.dev)
        side = torch.cuda.Stream()
        rc, r = self.ctx.select_and_gather(mode, gather_host, frac=frac, flags=flags, ids=ids,
                                           slots=slots, side_stream=side)
        if flags & K.KVS_GATHER_ASYNC:
            r = self.ctx.gather_counts()
        side.synchronize()
        torch.cuda.synchronize()
        res["rc"], res["gather"] = rc, r
        res["ids"] = [tuple(x) for x in ids.view(-1, 2)[: r.n_selected].cpu().tolist()]
        res["slots"] = slots[: r.n_selected].cpu().tolist()
        res["records"] = {sid: self.ctx.export_records(sid) for sid in self.ids
                          if not (flags & K.KVS_GATHER_DEMOTE)}
        if self.orc:
            res["oracle"] = self._oracle_step(q.cpu(), t)
        return res

    def _oracle_step(self, q, t):
        wl = self.wl
        outs, masses = {}, {}
        for s, sid in enumerate(self.ids):
            if sid not in self.orc:
                continue
            o = self.orc[sid]
            if self.kivi:      # whole groups behind the residual window are 2-bit
                Kf, Vf = O.kivi_effective(o.K, o.V)
                r = O.decode_with_mass(q[s], Kf, Vf, L=wl.L, Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d)
            elif self.fp8:     # the pages hold codes of the bf16 inputs
                kc, vc = self.seq_codes(sid, o)
                r = O.decode_with_mass(q[s], kc, vc, L=wl.L, Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d,
                                       k_lut=O.e4m3_lut(self.k_scale), v_lut=O.e4m3_lut(self.v_scale))
            else:
                r = O.decode_with_mass(q[s], o.K, o.V, L=wl.L, Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d)
            nb = len(o.rec)
            M = r["mass"]
            o.ambiguous |= np.abs(M * nb - 1.0) < TOUCH_MARGIN
            o.rec = O.score_update(o.rec, M, t, self.alpha, wl.recency_window, wl.weights, wl.cuts)
            outs[sid], masses[sid] = r["out"], M
        return {"out": outs, "mass": masses}

    # ------------------------------------------------------------------
    def excluded(self, sid):
        o = self.orc[sid]
        lo, hi = self.wl.cuts
        nearcut = (np.abs(o.rec["prio"] - lo) < CUT_MARGIN) | (np.abs(o.rec["prio"] - hi) < CUT_MARGIN)
        return nearcut | o.ambiguous

    def compare(self, res, check_records=True):
        """Asserts parity of one step; returns the error summary."""
        wl = self.wl
        summ = {"out_max_abs": 0.0, "mass_max_abs": 0.0, "score_max_abs": 0.0,
                "prio_max_abs": 0.0, "excluded": 0}
        orc = res["oracle"]
        out = res["out"].cpu().numpy()
        for s, sid in enumerate(self.ids):
            if sid not in self.orc:
                continue
            e = np.abs(out[s] - orc["out"][sid]).max()
            summ["out_max_abs"] = max(summ["out_max_abs"], float(e))
            slot = self.ctx.seq_info(sid)[0]
            nb = len(self.orc[sid].rec)
            gm = self.ctx.mass()[slot, :nb].cpu().numpy().astype(np.float64)
            summ["mass_max_abs"] = max(summ["mass_max_abs"], float(np.abs(gm - orc["mass"][sid]).max()))
            if not check_records:
                continue
            g = res["records"][sid]
            o = self.orc[sid].rec
            assert len(g) == len(o)
            assert np.array_equal(g["seq_id"], o["seq_id"]) and np.array_equal(g["block_idx"], o["block_idx"])
            summ["score_max_abs"] = max(summ["score_max_abs"], float(np.abs(g["score"] - o["score"]).max()))
            ex = self.excluded(sid)
            keep = ~ex
            summ["excluded"] += int(ex.sum())
            summ["prio_max_abs"] = max(summ["prio_max_abs"],
                                       float(np.abs(g["prio"][keep] - o["prio"][keep]).max(initial=0)))
            assert np.array_equal(g["tier"][keep], o["tier"][keep]), f"tier mismatch seq {sid}"
            assert np.array_equal(g["count"][keep], o["count"][keep]), f"count mismatch seq {sid}"
            assert np.array_equal(g["last_touch"][keep], o["last_touch"][keep])
            assert np.array_equal(g["lrfu"][keep], o["lrfu"][keep]), f"lrfu mismatch seq {sid}"
        assert summ["out_max_abs"] <= OUT_TOL, summ
        assert summ["mass_max_abs"] <= MASS_TOL, summ
        if check_records:
            assert summ["score_max_abs"] <= SCORE_TOL, summ
            assert summ["prio_max_abs"] <= SCORE_TOL, summ
        return summ

    def excluded_keys(self):
        out = set()
        for sid in self.tracked:
            ex = self.excluded(sid)
            out |= {(sid, int(b)) for b in np.nonzero(ex)[0]}
        return out

    def codes(self, Kb, Vb):
        return (O.quantize_bf16_e4m3(Kb, self.k_scale), O.quantize_bf16_e4m3(Vb, self.v_scale))

    def seq_codes(self, sid, o):
        """Codes of a sequence's tokens so far: tokens are write-once, so the
        codes of earlier steps are kept and only the new tokens quantised."""
        cache = self.__dict__.setdefault("_codes", {})
        kc, vc = cache.get(sid, (None, None))
        done = 0 if kc is None else kc.shape[0]
        if done < o.n:
            k_new, v_new = self.codes(o.K[done:], o.V[done:])
            kc = k_new if kc is None else np.concatenate([kc, k_new])
            vc = v_new if vc is None else np.concatenate([vc, v_new])
            cache[sid] = (kc, vc)
        return kc[:o.n], vc[:o.n]

    def oracle_page(self, sid, b):
        o = self.orc[sid]
        B = self.wl.block_tokens
        Kb, Vb = o.K[b * B:(b + 1) * B], o.V[b * B:(b + 1) * B]
        if self.fp8:
            return O.assemble_page(*self.codes(Kb, Vb), B)
        return O.assemble_page(Kb, Vb, B)

    def oracle_group_page(self, sid, grp):
        o = self.orc[sid]
        a = grp * O.KIVI_GROUP
        return O.kivi_group_page(o.K[a:a + O.KIVI_GROUP], o.V[a:a + O.KIVI_GROUP])

    def close(self):
        self.ctx.close()
