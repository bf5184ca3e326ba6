"""Runs a workload through the C ABI (CUDA path) and, beside it, through the
oracle, step by step, and compares them.

The oracle works in two modes:

 (i)  independent: attention output, block mass, scoring, tiers and
      selection computed from the inputs alone, for the sequences the oracle
      follows (all of them unless the run names a subset), at every step or
      at the steps the run names;
 (ii) conditioned scoring: the oracle's scoring, tiers, selection and gather
      plan fed the CUDA path's own fp32 block masses, for every sequence at
      every step, once those masses have been checked against mode (i)
      wherever mode (i) ran.  Both sides score in fp64 in the same operation
      order with no fused multiply-add, so mode (ii) must agree bit for bit
      in all 64 record bytes, in the selected id lists and in the gather plan
      (which page goes to which host slot), with no exclusion.

Mode (ii) is what makes the eviction lists checkable at sizes where mode (i)
cannot follow every sequence at every step; mode (i) is what pins the masses
it is fed.  Inputs for both sides come from the seeded generators in
``workloads`` (generated on the GPU, copied to the host for the oracle).

A run may hold several contexts ("lanes") fed identical inputs, one per
EMA weight alpha: attention and mass do not depend on alpha, so one oracle
attention pass serves every lane."""
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
CUT_MARGIN = 1e-5   # mode (i): records with oracle P this close to a cut are excluded
TOUCH_MARGIN = 1e-5 # mode (i): a touch decision the fp32 mass may flip (|M*nb - 1| below this)


def seq_ids_for(wl):
    # descending ids: call order differs from the ascending-id record order
    return [5000 - 17 * s for s in range(wl.nseq)]


@dataclass
class OracleSeq:
    """Mode (i) state of one followed sequence: its K/V on the host and, per
    lane, its independently scored records."""
    seq_id: int
    Kbuf: torch.Tensor            # host bf16 [capacity][L][Hkv][d]
    Vbuf: torch.Tensor
    n: int                        # tokens so far
    recs: list                    # per lane: oracle records, block order
    flips: list = None            # per lane: the path's touch decision differed at some step

    @property
    def K(self):
        return self.Kbuf[: self.n]

    @property
    def V(self):
        return self.Vbuf[: self.n]

    @property
    def rec(self):
        return self.recs[0]

    @rec.setter
    def rec(self, value):
        self.recs[0] = value


@dataclass
class Lane:
    """One context of the run, its EMA weight, and the mode (ii) records of
    every sequence (scored from this context's own masses)."""
    ctx: object
    alpha: float
    cond: dict = field(default_factory=dict)     # seq_id -> records (block order)


class Run:
    """oracle_seqs: indices of the sequences mode (i) follows (None = all);
    each sequence's attention, mass and records depend on it alone.
    attn_steps: the steps at which mode (i) attention runs (None = every
    step); mode (i) records are kept only when it runs at every step.
    alpha: one EMA weight, or a tuple of them (one context each).
    fused: each step decodes and scores in one call (kvs_decode_score_step)
    instead of kvs_decode_step + kvs_score_update."""

    def __init__(self, wl, alpha, *, staging_pages=8, chunk=4096, oracle_on=True,
                 oracle_seqs=None, attn_steps=None, pool_pages=None, extra_steps=0, device="cuda",
                 kv_dtype=K.KVS_KV_BF16, k_scale=1.0, v_scale=1.0, kivi_groups=0, fused=False):
        self.wl = wl
        self.fused = fused
        alphas = tuple(alpha) if isinstance(alpha, (tuple, list)) else (alpha,)
        self.alpha = alphas[0]
        self.dev = device
        self.ids = seq_ids_for(wl)
        self.mb = wl.max_blocks_per_seq() + (extra_steps + 15) // 16
        self.fp8 = kv_dtype == K.KVS_KV_FP8_E4M3
        self.kivi = kv_dtype == K.KVS_KV_KIVI2
        self.k_scale, self.v_scale = k_scale, v_scale
        self.lanes = []
        for a in alphas:
            cfg = K.make_config(wl.L, wl.Hq, wl.Hkv, wl.d, pool_pages or wl.pool_pages, max_seqs=wl.nseq,
                                max_blocks_per_seq=self.mb, alpha=a,
                                recency_window=wl.recency_window, weights=wl.weights, cuts=wl.cuts,
                                pool_seed=wl.seed, staging_pages=staging_pages, kv_dtype=kv_dtype,
                                k_scale=k_scale, v_scale=v_scale, kivi_groups=kivi_groups)
            self.lanes.append(Lane(K.Context(cfg), a))
        self.ctx = self.lanes[0].ctx
        self.oracle_on = oracle_on
        self.attn_steps = None if attn_steps is None else set(attn_steps)
        self.independent = oracle_on and attn_steps is None
        track = set(range(wl.nseq)) if oracle_seqs is None else set(oracle_seqs)
        self.tracked = [sid for s, sid in enumerate(self.ids) if oracle_on and s in track]
        self.t = 0
        self.ntok = list(wl.prefill_lens)
        self.orc = {}
        self.page_of = {}            # seq_id -> page identity per block (every sequence)
        B = wl.block_tokens
        pre_blocks = wl.shared_prefix_tokens // B
        cap_steps = wl.steps + extra_steps + 1
        for s, sid in enumerate(self.ids):
            n = wl.prefill_lens[s]
            if s > 0 and pre_blocks:
                for ln in self.lanes:
                    ln.ctx.seq_add(sid, self.ids[0], pre_blocks)
                start = wl.shared_prefix_tokens
            else:
                for ln in self.lanes:
                    ln.ctx.seq_add(sid)
                start = 0
            nb = (n + B - 1) // B
            self.page_of[sid] = [((0, b) if b < pre_blocks else (s, b)) for b in range(nb)]
            if oracle_on:
                for ln in self.lanes:
                    ln.cond[sid] = O.new_records(sid, 0, nb, 0)
            o = None
            if sid in self.tracked:
                shape = (n + cap_steps, wl.L, wl.Hkv, wl.d)
                o = OracleSeq(sid, torch.empty(shape, dtype=torch.bfloat16),
                              torch.empty(shape, dtype=torch.bfloat16), n,
                              [O.new_records(sid, 0, nb, 0) for _ in self.lanes],
                              [np.zeros(nb, bool) for _ in self.lanes])
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
                    kk, vv = Kt[lo:].contiguous(), Vt[lo:].contiguous()
                    for ln in self.lanes:
                        ln.ctx.append_tokens(sid, kk, vv)
                    del kk, vv
                del Kt, Vt
        torch.cuda.synchronize()

    # ------------------------------------------------------------------
    def step(self, gather_host=None, mode=K.KVS_SELECT_THRESH, flags=0, frac=0.0,
             batched_append=True):
        """One decode step over every sequence in every lane; returns a dict of
        GPU results (lane 0's at the top, every lane's under "lanes") and, if
        the oracle is on, the oracle's.  gather_host: the pinned host buffer
        of lane 0, or a list with one per lane.  batched_append: the new
        tokens go in through kvs_append_step (one call), else through one
        kvs_append_tokens call per sequence."""
        wl = self.wl
        B = wl.block_tokens
        self.t += 1
        t = self.t
        hosts = gather_host if isinstance(gather_host, (list, tuple)) else \
            [gather_host] + [None] * (len(self.lanes) - 1)
        new = [W.kv_tokens(wl, s, self.ntok[s], self.ntok[s] + 1, self.dev) for s in range(wl.nseq)]
        if batched_append:
            krow = torch.cat([k for k, _ in new]).contiguous()
            vrow = torch.cat([v for _, v in new]).contiguous()
            for ln in self.lanes:
                ln.ctx.append_step(self.ids, krow, vrow)
        for s, sid in enumerate(self.ids):
            n = self.ntok[s]
            Kt, Vt = new[s]
            if not batched_append:
                for ln in self.lanes:
                    ln.ctx.append_tokens(sid, Kt, Vt)
            if n % B == 0:          # a new block opens at the step counter t-1
                self.page_of[sid].append((s, n // B))
                if self.oracle_on:
                    for ln in self.lanes:
                        ln.cond[sid] = np.concatenate([ln.cond[sid], O.new_records(sid, n // B, 1, t - 1)])
            if sid in self.orc:
                o = self.orc[sid]
                if n % B == 0:
                    o.recs = [np.concatenate([r, O.new_records(sid, n // B, 1, t - 1)]) for r in o.recs]
                    o.flips = [np.append(f, False) for f in o.flips]
                o.Kbuf[n:n + 1].copy_(Kt.cpu())
                o.Vbuf[n:n + 1].copy_(Vt.cpu())
                o.n = n + 1
            self.ntok[s] = n + 1
        q = torch.stack([W.queries(wl, s, t, self.dev) for s in range(wl.nseq)]).contiguous()
        nrec = sum((n + B - 1) // B for n in self.ntok)
        lanes = []
        for ln, host in zip(self.lanes, hosts):
            ctx = ln.ctx
            out = torch.empty((wl.nseq, wl.L, wl.Hq, wl.d), dtype=torch.float32, device=self.dev)
            if self.fused:
                ctx.decode_score_step(self.ids, q, out)
            else:
                ctx.decode_step(self.ids, q, out)
                ctx.score_update()
            ids = torch.zeros(nrec * 2, dtype=torch.int64, device=self.dev)
            slots = torch.full((nrec,), -2, dtype=torch.int32, device=self.dev)
            side = torch.cuda.Stream()
            rc, r = ctx.select_and_gather(mode, host, frac=frac, flags=flags, ids=ids,
                                          slots=slots, side_stream=side)
            if flags & K.KVS_GATHER_ASYNC:
                r = ctx.gather_counts()
            side.synchronize()
            torch.cuda.synchronize()
            mass = ctx.mass().cpu().numpy()
            lr = {"out": out, "rc": rc, "gather": r, "host": host,
                  "ids": [tuple(x) for x in ids.view(-1, 2)[: r.n_selected].cpu().tolist()],
                  "slots": slots[: r.n_selected].cpu().tolist(),
                  "mass": {sid: mass[ctx.seq_info(sid)[0], :len(self.page_of[sid])].copy()
                           for sid in self.ids},
                  "records": {sid: ctx.export_records(sid) for sid in self.ids
                              if not (flags & K.KVS_GATHER_DEMOTE)}}
            lanes.append(lr)
        res = dict(lanes[0])
        res.update({"q": q, "lanes": lanes, "t": t, "mode": mode, "frac": frac, "flags": flags})
        if self.oracle_on:
            res["oracle"] = self._oracle_step(q.cpu(), t, lanes)
        return res

    def _oracle_step(self, q, t, lanes):
        wl = self.wl
        outs, masses = {}, {}
        attn = self.attn_steps is None or t in self.attn_steps
        for s, sid in enumerate(self.ids):
            if sid not in self.orc or not attn:
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
            # the touch rule M*nb >= 1 on the oracle's fp64 mass and on the
            # path's fp32 mass: a decision may differ only where the two
            # masses straddle the threshold within the mass tolerance
            for li, lr in enumerate(lanes):
                gm = lr["mass"][sid].astype(np.float64)
                flip = (gm * nb >= 1.0) != (M * nb >= 1.0)
                assert not np.any(flip & (np.abs(M * nb - 1.0) >= TOUCH_MARGIN)), \
                    f"t={t} seq {sid}: touch decision differs away from the threshold"
                o.flips[li] |= flip
            if self.independent:
                o.recs = [O.score_update(rec, M, t, ln.alpha, wl.recency_window, wl.weights, wl.cuts)
                          for rec, ln in zip(o.recs, self.lanes)]
            outs[sid], masses[sid] = r["out"], M
        # mode (ii): every sequence scored from the lane's own fp32 masses
        for ln, lr in zip(self.lanes, lanes):
            for sid in self.ids:
                gm = lr["mass"][sid].astype(np.float64)
                ln.cond[sid] = O.score_update(ln.cond[sid], gm, t, ln.alpha, wl.recency_window,
                                              wl.weights, wl.cuts)
        return {"out": outs, "mass": masses, "attn": attn}

    # ------------------------------------------------------------------
    def near_cut(self, sid, lane=0):
        rec = self.orc[sid].recs[lane]
        lo, hi = self.wl.cuts
        return (np.abs(rec["prio"] - lo) < CUT_MARGIN) | (np.abs(rec["prio"] - hi) < CUT_MARGIN)

    def excluded(self, sid, lane=0):
        """Mode (i) exclusion: records whose oracle P lies within CUT_MARGIN
        of a cut, and records whose touch decision went the other way on the
        path's fp32 mass at some step (possible only within TOUCH_MARGIN of
        the threshold, asserted when it happens; counted as touch_flips).
        Mode (ii) compares every record, these included, bit for bit."""
        return self.near_cut(sid, lane) | self.orc[sid].flips[lane]

    def compare(self, res, check_records=True):
        """Asserts parity of one step in every lane; returns the error summary.

        Mode (i): output and mass of the followed sequences against the
        independent oracle (where its attention ran); their records against
        the independent scoring (when it runs at every step), tiers, counts,
        touch times and LRFU scores bit-exact outside the cut exclusion.
        Mode (ii): the 64 bytes of every record of every sequence, the id
        list and the gather plan bit for bit against the conditioned oracle."""
        summ = {"out_max_abs": 0.0, "mass_max_abs": 0.0, "mass_sum_dev": 0.0, "score_max_abs": 0.0,
                "prio_max_abs": 0.0, "excluded_near_cut": 0, "touch_flips": 0,
                "cond_records": 0, "cond_ids": 0}
        orc = res["oracle"]
        for li, (ln, lr) in enumerate(zip(self.lanes, res["lanes"])):
            # the masses mode (ii) is fed: per-sequence sums (any size), then mode (i)
            for sid in self.ids:
                m = lr["mass"][sid].astype(np.float64)
                assert np.all(m >= 0.0) and np.all(np.isfinite(m)), sid
                summ["mass_sum_dev"] = max(summ["mass_sum_dev"], abs(float(m.sum()) - 1.0))
            assert summ["mass_sum_dev"] <= MASS_TOL, summ
            if orc["attn"]:
                out = lr["out"].cpu().numpy()
                for s, sid in enumerate(self.ids):
                    if sid not in orc["out"]:
                        continue
                    e = np.abs(out[s] - orc["out"][sid]).max()
                    summ["out_max_abs"] = max(summ["out_max_abs"], float(e))
                    gm = lr["mass"][sid].astype(np.float64)
                    summ["mass_max_abs"] = max(summ["mass_max_abs"],
                                               float(np.abs(gm - orc["mass"][sid]).max()))
            if check_records and lr["records"]:
                # mode (ii): every byte of every record
                for sid in self.ids:
                    g = lr["records"][sid]
                    c = ln.cond[sid]
                    assert len(g) == len(c), sid
                    if g.tobytes() != c.tobytes():
                        bad = np.nonzero(g.view(np.uint8).reshape(-1, 64) != c.view(np.uint8).reshape(-1, 64))
                        raise AssertionError(f"lane {li} t={res['t']} seq {sid}: conditioned records differ "
                                             f"at block {int(bad[0][0])} byte {int(bad[1][0])}")
                    summ["cond_records"] += len(c)
            if check_records and self.independent and lr["records"]:
                for sid in self.tracked:
                    g = lr["records"][sid]
                    o = self.orc[sid].recs[li]
                    assert len(g) == len(o)
                    assert np.array_equal(g["seq_id"], o["seq_id"]) and np.array_equal(g["block_idx"], o["block_idx"])
                    summ["score_max_abs"] = max(summ["score_max_abs"], float(np.abs(g["score"] - o["score"]).max()))
                    keep = ~self.excluded(sid, li)
                    summ["excluded_near_cut"] += int(self.near_cut(sid, li).sum())
                    summ["touch_flips"] += int(self.orc[sid].flips[li].sum())
                    summ["prio_max_abs"] = max(summ["prio_max_abs"],
                                               float(np.abs(g["prio"][keep] - o["prio"][keep]).max(initial=0)))
                    assert np.array_equal(g["tier"][keep], o["tier"][keep]), f"tier mismatch seq {sid}"
                    assert np.array_equal(g["count"][keep], o["count"][keep]), f"count mismatch seq {sid}"
                    assert np.array_equal(g["last_touch"][keep], o["last_touch"][keep])
                    assert np.array_equal(g["lrfu"][keep], o["lrfu"][keep]), f"lrfu mismatch seq {sid}"
            summ["cond_ids"] += self._check_list(ln, lr, res)
        assert summ["out_max_abs"] <= OUT_TOL, summ
        assert summ["mass_max_abs"] <= MASS_TOL, summ
        if check_records:
            assert summ["score_max_abs"] <= SCORE_TOL, summ
            assert summ["prio_max_abs"] <= SCORE_TOL, summ
        return summ

    def cond_list(self, lane, mode, frac):
        """The conditioned oracle's selection in `lane`."""
        ln = self.lanes[lane] if isinstance(lane, int) else lane
        if mode == K.KVS_SELECT_THRESH:
            return O.select_thresh(ln.cond)
        if mode == K.KVS_SELECT_LOWFRAC:
            return O.select_lowfrac(ln.cond, frac)
        return O.select_lrfu(ln.cond, frac, ln.alpha)

    def cond_plan(self, ids):
        """Pages the conditioned oracle gathers for a list: identities in order."""
        refs = {}
        for sid in self.ids:
            for b, pid in enumerate(self.page_of[sid]):
                refs.setdefault(pid, set()).add((sid, b))
        page_of = {(sid, b): pid for sid in self.ids for b, pid in enumerate(self.page_of[sid])}
        return O.gather_plan(ids, page_of, refs), page_of

    def _check_list(self, ln, lr, res):
        """Mode (ii): the id list bit for bit; the eligibility of each listed
        page and, in list mode, its host slot (the plan position, -1 past a
        truncated buffer).  Returns the list length."""
        want = self.cond_list(ln, res["mode"], res["frac"])
        assert lr["ids"] == want, f"t={res['t']}: id list differs from the conditioned oracle " \
                                  f"({len(lr['ids'])} vs {len(want)} ids)"
        if self.kivi or lr["gather"].n_selected == 0 or res["flags"] & K.KVS_GATHER_DEMOTE:
            return len(want)
        plan, page_of = self.cond_plan(want)
        assert lr["gather"].n_pages == len(plan)
        pos = {p: i for i, p in enumerate(plan)}
        mirror = bool(res["flags"] & K.KVS_GATHER_MIRROR)
        host = lr["host"]
        cap = 0 if host is None else host.numel() // ln.ctx.page_bytes
        for key, slot in zip(lr["ids"], lr["slots"]):
            i = pos.get(page_of[key])
            if mirror:
                assert (slot >= 0) == (i is not None), key
            elif host is not None:
                assert slot == (i if i is not None and i < cap else -1), (key, slot, i)
        return len(want)

    def excluded_keys(self, lane=0):
        out = set()
        for sid in self.tracked:
            ex = self.excluded(sid, lane)
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
        for ln in self.lanes:
            ln.ctx.close()
