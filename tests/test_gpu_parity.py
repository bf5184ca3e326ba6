"""Parity of the CUDA path (through the C ABI) with the fp64 oracle."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import paged_kv_cache_flash_gb300 as K
import workloads as W
from gpu_harness import Run, seq_ids_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_flash_gb300 import build
    build.build()


def _pinned(nbytes):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8).pin_memory()


def _check_gather(run, res, host, sample=None, lane=0):
    """The id list, each listed page's eligibility (the reference-count rule)
    and its host slot are checked bit for bit against the conditioned oracle
    by run.compare.  Here: the independent oracle's list over the followed
    sequences (outside the cut exclusion), and the bytes of every gathered
    page of a followed sequence (a seeded sample of `sample` of them if
    given) against the oracle's page assembly.  Returns the pages compared."""
    lr = res["lanes"][lane]
    if run.independent:
        excl = run.excluded_keys(lane)
        tracked = set(run.tracked)
        orc_ids = O.select_thresh({sid: run.orc[sid].recs[lane] for sid in run.tracked})
        got = [k for k in lr["ids"] if k[0] in tracked]
        assert [k for k in got if k not in excl] == [k for k in orc_ids if k not in excl]
    assert lr["ids"] == sorted(lr["ids"])
    pb = run.lanes[lane].ctx.page_bytes
    hb = host.numpy()
    pairs = [(k, s) for k, s in zip(lr["ids"], lr["slots"]) if k[0] in run.orc and s >= 0]
    if sample is not None and sample < len(pairs):
        pick = sorted(np.random.default_rng(11 + res["t"]).choice(len(pairs), sample, replace=False))
        pairs = [pairs[j] for j in pick]
    for (sid, b), slot in pairs:
        assert hb[slot * pb:(slot + 1) * pb].tobytes() == run.oracle_page(sid, b), (sid, b)
    return len(pairs)


def test_tiny_end_to_end():
    """Tiny workload: 2 layers, 4:1 GQA, d=64, 1 x 256 tokens, 4 steps."""
    wl = W.workload("tiny")
    run = Run(wl, wl.alphas[0])
    host = _pinned(wl.pool_pages * wl.page_bytes)
    for _ in range(wl.steps):
        res = run.step(host)
        summ = run.compare(res)
        _check_gather(run, res, host)
        assert res["rc"] == K.KVS_OK
    run.ctx.check_device()
    print("tiny", summ)
    run.close()


def test_ragged_multi_sequence_and_shared_prefix():
    """Three sequences of ragged lengths (1 token .. 9 blocks + tail), two of
    them sharing the first 2 blocks of the first (refcounted pages)."""
    wl = W.workload("tiny", prefill_lens=(40, 33, 150), shared_prefix_tokens=32,
                    pool_pages=40, steps=20, skew=True)
    run = Run(wl, 0.3)
    host = _pinned(wl.pool_pages * wl.page_bytes)
    for i in range(wl.steps):
        # alternate the batched append and the per-sequence one
        res = run.step(host, batched_append=bool(i % 2))
        run.compare(res)
        _check_gather(run, res, host)
    # the shared pages are gathered only when all three users list them
    run.close()


@pytest.mark.parametrize("nseq,max_len", [(80, 500), (K.KVS_MAX_CALL_SEQS, 140)])
def test_many_sequences_ring_uploads_and_multi_tile_selection(nseq, max_len):
    """80 sequences of 1..499 tokens, and the most one call takes (256) of
    1..139 tokens, in every call: the decode set (more than 63 entries) and the
    step append (more than 16) travel through the upload ring instead of
    kernel parameters, and the 1,000+ records take the two-kernel (count,
    then scatter) selection; 3 steps against the full oracle, listed ids and
    gathered pages checked."""
    rng = np.random.default_rng(0x6B76 + nseq)
    lens = tuple(int(x) for x in rng.integers(1, max_len, size=nseq))
    pool = sum((n + 4 + 15) // 16 for n in lens) + 8
    wl = W.workload("tiny", prefill_lens=lens, pool_pages=pool, steps=3, skew=True)
    assert sum((n + wl.steps + 15) // 16 for n in lens) > 1024
    run = Run(wl, 0.15)
    host = _pinned(pool * wl.page_bytes)
    for _ in range(wl.steps):
        res = run.step(host)
        summ = run.compare(res)
        _check_gather(run, res, host)
    run.ctx.check_device()
    print(nseq, "sequences", summ)
    run.close()


@pytest.mark.parametrize("name,kw", [
    ("tiny", dict(prefill_lens=(40, 33, 150), shared_prefix_tokens=32, pool_pages=40, steps=6, skew=True)),
    ("l70b_8k", dict(L=6, prefill_lens=(3000, 1, 700), pool_pages=300, steps=4))])
def test_fused_decode_score_matches_two_calls(name, kw):
    """kvs_decode_score_step (scores in the decode epilogue) against
    kvs_decode_step + kvs_score_update on a second context fed the same
    steps: outputs, masses, all record bytes and the lists bit for bit, the
    fused side also against the oracle; a score update after a fused step is
    refused."""
    wl = W.workload(name, **kw)
    two, one = Run(wl, 0.15, oracle_on=False), Run(wl, 0.15, fused=True)
    for _ in range(wl.steps):
        a, b = two.step(None), one.step(None)
        one.compare(b)
        assert torch.equal(a["out"], b["out"])
        assert all(np.array_equal(a["mass"][s], b["mass"][s]) for s in two.ids)
        assert all(a["records"][s].tobytes() == b["records"][s].tobytes() for s in two.ids)
        assert a["ids"] == b["ids"]
    with pytest.raises(K.KvsError) as e:
        one.ctx.score_update()
    assert e.value.code == K.KVS_EINVAL
    one.ctx.check_device()
    two.close()
    one.close()


def test_single_token_sequence_and_large_group():
    """One-token sequences (nothing but block 0) and the full 8:1 group at d=128."""
    wl = W.workload("l70b_8k", L=3, prefill_lens=(1, 17), pool_pages=8, steps=3)
    run = Run(wl, 0.15)
    for _ in range(wl.steps):
        res = run.step(None, batched_append=False)
        run.compare(res)
    run.close()


def test_llama70b_shape_cut():
    """All 80 layers, 64/8 heads, d=128, one ragged 1,000-token sequence."""
    wl = W.workload("l70b_8k", prefill_lens=(1000,), pool_pages=70, steps=2)
    run = Run(wl, 0.15)
    host = _pinned(64 * wl.page_bytes)
    for _ in range(wl.steps):
        res = run.step(host)
        summ = run.compare(res)
        _check_gather(run, res, host)
    print("l70b cut", summ)
    run.close()


@pytest.mark.parametrize("fmt,Hq,Hkv,d", [
    ("bf16", 4, 4, 64), ("bf16", 6, 2, 128), ("bf16", 16, 2, 64), ("bf16", 8, 4, 128),
    ("fp8", 4, 4, 128), ("fp8", 6, 2, 128), ("kivi2", 8, 4, 128), ("kivi2", 3, 3, 128)])
def test_geometry_matrix(fmt, Hq, Hkv, d):
    """GQA groups of 1, 2, 3 and 8 query heads at head dims 64 and 128 in
    every page format the geometry allows: 3 layers, a one-token sequence, a
    mid-block tail and a multi-chunk sequence, both append paths."""
    wl = W.workload("l70b_8k", L=3, Hq=Hq, Hkv=Hkv, d=d, prefill_lens=(1, 200, 777),
                    pool_pages=80, steps=3)
    kw = {}
    if fmt == "fp8":
        kw = dict(kv_dtype=K.KVS_KV_FP8_E4M3, k_scale=0.5, v_scale=2.0)
    elif fmt == "kivi2":
        kw = dict(kv_dtype=K.KVS_KV_KIVI2, kivi_groups=40)
    run = Run(wl, 0.15, **kw)
    host = None if fmt == "kivi2" else _pinned(wl.pool_pages * run.ctx.page_bytes)
    if fmt == "kivi2":
        assert _check_kivi_groups(run) == (64 + 640) // 32
    for i in range(wl.steps):
        res = run.step(host, batched_append=bool(i % 2))
        summ = run.compare(res)
        if host is not None:
            _check_gather(run, res, host)
    run.ctx.check_device()
    print(fmt, Hq, Hkv, d, summ)
    run.close()


# ------------------------------------------------------------- FP8 pages


@pytest.mark.parametrize("scales", [(1.0, 1.0), (0.5, 0.25)])
def test_fp8_pages_parity(scales):
    """FP8 E4M3 pages: codes quantised on append (bit-exact against the
    oracle's quantiser, checked through the gathered page bytes), decode over
    the codes within the bf16 tolerances, two append paths, ragged lengths."""
    wl = W.workload("l70b_8k", L=4, prefill_lens=(300, 1000, 17), pool_pages=100, steps=4)
    run = Run(wl, 0.15, kv_dtype=K.KVS_KV_FP8_E4M3, k_scale=scales[0], v_scale=scales[1])
    assert run.ctx.page_bytes == wl.page_bytes // 2
    host = _pinned(wl.pool_pages * run.ctx.page_bytes)
    for i in range(wl.steps):
        res = run.step(host, batched_append=bool(i % 2))
        summ = run.compare(res)
        _check_gather(run, res, host)
    run.ctx.check_device()
    print("fp8", scales, summ)
    run.close()


def test_fp8_demote_prefetch_round_trip():
    """FP8 pages (half size) through demotion to pinned host and back by a
    budgeted prefetch: code pages byte-equal, records restored, decoding
    resumes in parity."""
    wl = W.workload("l70b_8k", L=2, prefill_lens=(400, 700), pool_pages=90, steps=4)
    run = Run(wl, 0.05, kv_dtype=K.KVS_KV_FP8_E4M3, k_scale=0.5, v_scale=0.5)
    for _ in range(2):
        run.compare(run.step(None))
    before = {sid: run.ctx.export_records(sid) for sid in run.ids}
    pages = {(sid, b): run.ctx.page_bytes_of(p).cpu().numpy().tobytes()
             for sid in run.ids for b, p in enumerate(run.ctx.seq_info(sid)[3])}
    nrec = sum(len(v) for v in before.values())
    host = _pinned(nrec * run.ctx.page_bytes)
    ids = torch.zeros(2 * nrec, dtype=torch.int64, device="cuda")
    rc, r = run.ctx.select_and_gather(K.KVS_SELECT_LOWFRAC, host, frac=0.3,
                                      flags=K.KVS_GATHER_DEMOTE, ids=ids)
    torch.cuda.synchronize()
    assert rc == K.KVS_OK and r.n_demoted == r.n_selected == O.lowfrac_k(nrec, 0.3)
    got = [tuple(x) for x in ids.view(-1, 2)[: r.n_demoted].cpu().tolist()]
    pb = run.ctx.page_bytes
    for i, key in enumerate(got):
        assert host.numpy()[i * pb:(i + 1) * pb].tobytes() == pages[key] == run.oracle_page(*key)
    side = torch.cuda.Stream()
    while run.ctx.prefetch_plan(1):
        run.ctx.prefetch(10, host, stream=side)
    side.synchronize()
    for sid in run.ids:
        assert run.ctx.export_records(sid).tobytes() == before[sid].tobytes()
        for b, p in enumerate(run.ctx.seq_info(sid)[3]):
            assert run.ctx.page_bytes_of(p).cpu().numpy().tobytes() == pages[(sid, b)]
    for _ in range(2):
        run.compare(run.step(None))
    run.close()


def test_fp8_config_checks():
    with pytest.raises(K.KvsError):
        K.kvs_required_sizes(K.make_config(2, 8, 2, 64, 17, 1, 18, kv_dtype=K.KVS_KV_FP8_E4M3))
    with pytest.raises(K.KvsError):
        K.kvs_required_sizes(K.make_config(2, 16, 2, 128, 17, 1, 18, kv_dtype=K.KVS_KV_FP8_E4M3,
                                           k_scale=0.0))


# ------------------------------------------------------------ KIVI 2-bit


def _check_kivi_groups(run, sample=None):
    """Every quantised group: both blocks name one group page whose bytes are
    the oracle's quantisation in the tile layout (on a seeded sample of
    `sample` groups per sequence if given); the rest are bf16 pages."""
    rng = np.random.default_rng(5)
    n_groups = 0
    for sid in run.tracked:
        _, ntok, nb, table = run.ctx.seq_info(sid)
        q = O.kivi_quantized_tokens(ntok)
        for b, p in enumerate(table):
            if b < q // 16:
                assert p <= -2 and table[b ^ 1] == p, (sid, b, p)
            else:
                assert p >= 0, (sid, b, p)
        n_groups += q // 32
        check = range(q // 32)
        if sample is not None and sample < q // 32:
            check = sorted(rng.choice(q // 32, sample, replace=False))
        for grp in check:
            gp = -2 - table[2 * grp]
            got = run.ctx.group_bytes_of(gp).cpu().numpy().tobytes()
            assert got == run.oracle_group_page(sid, grp), (sid, grp)
    return n_groups


def test_kivi_parity():
    """2-bit groups behind a 128-token residual window: group pages equal the
    oracle's quantisation byte for byte; decode over groups + residual pages
    matches the oracle on the effective values while sequences cross group
    boundaries, through both append paths; selection returns ids only."""
    wl = W.workload("l70b_8k", L=3, prefill_lens=(300, 1000, 17, 477), pool_pages=140, steps=40)
    run = Run(wl, 0.15, kv_dtype=K.KVS_KV_KIVI2, kivi_groups=64)
    assert _check_kivi_groups(run) == (160 + 864 + 0 + 320) // 32
    for i in range(wl.steps):
        res = run.step(None, batched_append=bool(i % 2))
        summ = run.compare(res)
        if i % 13 == 0:         # the THRESH list (ids only in 2-bit contexts)
            excl = run.excluded_keys()
            got = [k for k in res["ids"] if k not in excl]
            assert got == [k for k in O.select_thresh({s: run.orc[s].rec for s in run.ids}) if k not in excl]
            assert res["gather"].n_pages == 0
    n = _check_kivi_groups(run)
    assert n == (192 + 896 + 0 + 384) // 32
    # LOWFRAC and LRFU victims as id lists (ids only in 2-bit contexts): the
    # oracle's selection over the device's records (compared above)
    recs = {s: run.ctx.export_records(s) for s in run.ids}
    nrec = sum(len(v) for v in recs.values())
    ids = torch.zeros(2 * nrec, dtype=torch.int64, device="cuda")
    for mode, ref in ((K.KVS_SELECT_LOWFRAC, O.select_lowfrac(recs, 0.2)),
                      (K.KVS_SELECT_LRFU, O.select_lrfu(recs, 0.2, 0.15))):
        rc, r = run.ctx.select_and_gather(mode, frac=0.2, ids=ids)
        assert rc == K.KVS_OK and r.n_pages == 0
        assert [tuple(x) for x in ids.view(-1, 2)[: r.n_selected].cpu().tolist()] == ref
    run.ctx.check_device()
    print("kivi", summ, n, "groups")
    run.close()


def test_kivi_error_paths():
    wl = W.workload("l70b_8k", L=2, prefill_lens=(300,), pool_pages=40, steps=2)
    cfg = K.make_config(wl.L, wl.Hq, wl.Hkv, wl.d, 40, 2, 40, kv_dtype=K.KVS_KV_KIVI2, kivi_groups=4)
    ctx = K.Context(cfg)
    Kt, Vt = W.kv_tokens(wl, 0, 0, 300, "cuda")
    ctx.seq_add(1)
    with pytest.raises(K.KvsError) as e:          # 300 tokens need 5 groups: nothing appended
        ctx.append_tokens(1, Kt, Vt)
    assert e.value.code == K.KVS_ENOMEM and ctx.seq_info(1)[1] == 0
    ctx.append_tokens(1, Kt[:200].contiguous(), Vt[:200].contiguous())    # 2 groups
    _, ntok, nb, t = ctx.seq_info(1)
    assert ntok == 200 and nb == 13
    assert t[0] == t[1] <= -2 and t[2] == t[3] <= -2 and t[0] != t[2] and min(t[4:]) >= 0
    with pytest.raises(K.KvsError) as e:          # no shared blocks in 2-bit contexts
        ctx.seq_add(2, 1, 2)
    assert e.value.code == K.KVS_EINVAL
    q = torch.zeros((1, wl.L, wl.Hq, wl.d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((1, wl.L, wl.Hq, wl.d), device="cuda")
    ctx.decode_step([1], q, out)
    ctx.score_update()
    host = _pinned(4 * ctx.page_bytes)
    with pytest.raises(K.KvsError) as e:          # no gathers of group pages
        ctx.select_and_gather(K.KVS_SELECT_THRESH, host)
    assert e.value.code == K.KVS_EINVAL
    free = ctx.free_pages()
    ctx.seq_remove(1)
    assert ctx.free_pages() == free + (200 - 64 + 15) // 16
    ctx.check_device()
    ctx.close()


# --------------------------------------------------------------- scoring


def _mass_tensor(run, masses):
    m = torch.zeros((len(run.ids), run.mb), dtype=torch.float32)
    for i, sid in enumerate(run.ids):
        m[i, :len(masses[sid])] = torch.from_numpy(masses[sid])
    return m.cuda()


@pytest.mark.parametrize("alpha,cuts", [(0.15, (0.3, 0.6)), (1.0, (0.3, 0.6)),
                                        (0.0, (0.25, 0.25 + 0.2))])
def test_scoring_bit_exact_on_injected_mass(alpha, cuts):
    """Scoring, tiers and both selections driven from the same seeded masses
    on both sides must agree bit for bit in all 64 record bytes.  With
    alpha = 0 and cuts (0.25, 0.25+0.2) every touched interior block sits
    exactly on cut_lo and every touched anchor exactly on cut_hi."""
    cuts = (cuts[0], float(np.float64(0.25) + np.float64(0.2))) if alpha == 0.0 else cuts
    wl = W.workload("tiny", prefill_lens=(37, 300, 1), pool_pages=40, cuts=cuts, steps=0)
    run = Run(wl, alpha)
    rng = np.random.default_rng(7)
    seen = set()
    for t in range(1, 90):
        masses = {}
        for sid in run.ids:
            nb = len(run.orc[sid].rec)
            m = W.synthetic_masses(1000 * t + sid, nb)
            m[rng.random(nb) < (0.6 if t < 70 else 1.0)] = 0.0   # long silences: R clips
            masses[sid] = m
        run.ctx.debug_advance(1)
        run.ctx.debug_set_mass(run.ids, _mass_tensor(run, masses))
        run.ctx.score_update()
        for sid in run.ids:
            o = run.orc[sid]
            o.rec = O.score_update(o.rec, masses[sid].astype(np.float64), t, alpha,
                                   wl.recency_window, wl.weights, wl.cuts)
            g = run.ctx.export_records(sid)
            assert g.tobytes() == o.rec.tobytes(), f"t={t} seq={sid}"
            seen |= set(o.rec["tier"].tolist())
        if t % 10 == 0:
            recs = {sid: run.orc[sid].rec for sid in run.ids}
            _, r = run.ctx.select_and_gather(K.KVS_SELECT_THRESH)
            assert r.n_selected == len(O.select_thresh(recs))
            ids = torch.zeros(2 * 400, dtype=torch.int64, device="cuda")
            _, r = run.ctx.select_and_gather(K.KVS_SELECT_LOWFRAC, frac=0.25, ids=ids)
            got = [tuple(x) for x in ids.view(-1, 2)[: r.n_selected].cpu().tolist()]
            assert got == O.select_lowfrac(recs, 0.25)
            if alpha < 1.0:     # LRFU victims: key order and the brute-force audit
                _, r = run.ctx.select_and_gather(K.KVS_SELECT_LRFU, frac=0.25, ids=ids)
                got = [tuple(x) for x in ids.view(-1, 2)[: r.n_selected].cpu().tolist()]
                assert got == O.select_lrfu(recs, 0.25, alpha)
                assert got == O.lrfu_victims_brute_force(recs, 0.25, t, alpha)
    if alpha == 0.0:     # blocks sat exactly on both cuts at some step
        assert {0, 1, 2} <= seen
    run.close()


def test_lrfu_near_tie_keys_order_like_the_oracle():
    """Planted records whose LRFU keys tie up to rounding ([RETR] s.3: a
    block touched at t with score S and one touched at t + d with score
    S*(1-alpha)^d have the same key): the device's victim lists equal the
    oracle's bit for bit, because both take the key's logarithms by the same
    fixed sequence of fp64 operations."""
    alpha = 0.15
    wl = W.workload("tiny", prefill_lens=(500, 700, 300), pool_pages=120, steps=1, skew=True)
    run = Run(wl, alpha)
    run.compare(run.step(None))              # a decode set and its records
    rng = np.random.default_rng(31)
    planted = {}
    for sid in run.ids:
        r = run.ctx.export_records(sid)
        n = len(r)
        d = rng.integers(0, 60, n)
        S0 = np.where(rng.random(n) < 0.5, 0.9, 0.3)         # two clusters of keys
        r["lrfu"] = S0 * O.lrfu_decay(alpha, d)
        r["last_touch"] = (20 + d).astype(np.uint64)
        r["lrfu"][rng.random(n) < 0.05] = 0.0                 # never touched: key -inf
        run.ctx.debug_import_records(sid, r)
        planted[sid] = r
    allr = np.concatenate([planted[s] for s in sorted(planted)])
    key = O.lrfu_key(allr["lrfu"], allr["last_touch"], alpha)
    c = O.lrfu_slope(alpha)
    near = [np.abs(key - (np.log(S0) + 20 * c)) < 1e-12 for S0 in (0.9, 0.3)]
    assert np.all(near[0] | near[1] | np.isneginf(key))
    # each cluster: keys equal up to rounding, yet not all equal
    assert all(near_c.sum() > 20 and len(np.unique(key[near_c])) > 1 for near_c in near)
    nrec = len(allr)
    ids = torch.zeros(2 * nrec, dtype=torch.int64, device="cuda")
    for frac in (0.1, 0.3, 0.5, 0.7):
        rc, r = run.ctx.select_and_gather(K.KVS_SELECT_LRFU, frac=frac, ids=ids)
        got = [tuple(x) for x in ids.view(-1, 2)[: r.n_selected].cpu().tolist()]
        assert got == O.select_lrfu(planted, frac, alpha), frac
    run.close()


# ------------------------------------------------------ demote / readmit


def test_demote_readmit_round_trip():
    """LOWFRAC 10 % demotion to pinned host, then re-admission into other
    pages: pages byte-equal, records restored bit for bit, decoding after
    the round trip still matches the oracle."""
    wl = W.workload("tiny", prefill_lens=(200, 333, 97, 150), pool_pages=60, steps=6, skew=True)
    run = Run(wl, 0.05)
    for _ in range(3):
        run.compare(run.step(None))
    before = {sid: run.ctx.export_records(sid) for sid in run.ids}
    tables = {sid: run.ctx.seq_info(sid)[3] for sid in run.ids}
    pages_before = {}
    for sid in run.ids:
        for b, p in enumerate(tables[sid]):
            pages_before[(sid, b)] = run.ctx.page_bytes_of(p).cpu().numpy().tobytes()
    nrec = sum(len(v) for v in before.values())
    host = _pinned(nrec * run.ctx.page_bytes)
    ids = torch.zeros(2 * nrec, dtype=torch.int64, device="cuda")
    free0 = run.ctx.free_pages()
    rc, r = run.ctx.select_and_gather(K.KVS_SELECT_LOWFRAC, host, frac=0.10,
                                      flags=K.KVS_GATHER_DEMOTE, ids=ids)
    torch.cuda.synchronize()
    assert rc == K.KVS_OK
    k = int(np.floor(0.10 * nrec))
    assert r.n_selected == k == r.n_demoted
    got = [tuple(x) for x in ids.view(-1, 2)[:k].cpu().tolist()]
    assert got == O.select_lowfrac(before, 0.10)
    assert run.ctx.free_pages() == free0 + k
    hb = host.numpy()
    pb = run.ctx.page_bytes
    for i, key in enumerate(got):
        assert hb[i * pb:(i + 1) * pb].tobytes() == pages_before[key]
        assert run.ctx.seq_info(key[0])[3][key[1]] == -1
    q = torch.zeros((wl.nseq, wl.L, wl.Hq, wl.d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((wl.nseq, wl.L, wl.Hq, wl.d), device="cuda")
    with pytest.raises(K.KvsError) as e:       # blocks are missing: refused
        run.ctx.decode_step(run.ids, q, out)
    assert e.value.code == K.KVS_EINVAL
    run.ctx.readmit(got, host)
    torch.cuda.synchronize()
    for sid in run.ids:
        assert run.ctx.export_records(sid).tobytes() == before[sid].tobytes()
        for b, p in enumerate(run.ctx.seq_info(sid)[3]):
            assert run.ctx.page_bytes_of(p).cpu().numpy().tobytes() == pages_before[(sid, b)]
    with pytest.raises(K.KvsError) as e:
        run.ctx.readmit(got[:1], host)
    assert e.value.code == K.KVS_EEXIST
    for _ in range(2):                          # decoding resumes in parity
        run.compare(run.step(None))
    run.close()


def test_prefetch_order_and_readmission():
    """Demote half of the blocks, then: the device fetch order equals the
    oracle's (keys, classes, blends bit for bit) for several budgets; a
    budgeted prefetch re-admits exactly the plan's head with pages and
    records restored; the rest follows; decoding resumes in parity."""
    wl = W.workload("tiny", prefill_lens=(700, 1333, 420, 950), pool_pages=240, steps=5, skew=True)
    run = Run(wl, 0.05)
    for _ in range(3):
        run.compare(run.step(None))
    before = {sid: run.ctx.export_records(sid) for sid in run.ids}
    pages_before = {}
    for sid in run.ids:
        for b, p in enumerate(run.ctx.seq_info(sid)[3]):
            pages_before[(sid, b)] = run.ctx.page_bytes_of(p).cpu().numpy().tobytes()
    nrec = sum(len(v) for v in before.values())
    host = _pinned(nrec * run.ctx.page_bytes)
    ids = torch.zeros(2 * nrec, dtype=torch.int64, device="cuda")
    rc, r = run.ctx.select_and_gather(K.KVS_SELECT_LOWFRAC, host, frac=0.5,
                                      flags=K.KVS_GATHER_DEMOTE, ids=ids)
    torch.cuda.synchronize()
    assert rc == K.KVS_OK and r.n_demoted == r.n_selected
    demoted = [tuple(x) for x in ids.view(-1, 2)[: r.n_demoted].cpu().tolist()]
    ntok = {sid: run.ctx.seq_info(sid)[1] for sid in run.ids}
    score = {(sid, int(b)): float(e) for sid in run.ids
             for b, e in zip(before[sid]["block_idx"], before[sid]["score"])}

    def oracle_plan(keys, budget):
        return O.prefetch_order([(s, b, ntok[s], score[(s, b)]) for s, b in keys], budget)

    full = oracle_plan(demoted, len(demoted))
    assert {c for _, _, c, _ in full} == {0, 1, 2}, "the case must cover every class"
    for budget in (1, 7, 64, len(demoted), K.KVS_PREFETCH_MAX):
        assert run.ctx.prefetch_plan(budget) == oracle_plan(demoted, budget)
    side = torch.cuda.Stream()
    head = run.ctx.prefetch(20, host, stream=side)
    side.synchronize()
    assert head == full[:20]
    for s, b, _, _ in head:
        p = run.ctx.seq_info(s)[3][b]
        assert p >= 0 and run.ctx.page_bytes_of(p).cpu().numpy().tobytes() == pages_before[(s, b)]
    rest = [k for k in demoted if k not in {(s, b) for s, b, _, _ in head}]
    assert run.ctx.prefetch_plan(K.KVS_PREFETCH_MAX) == oracle_plan(rest, len(rest))
    tail = run.ctx.prefetch(K.KVS_PREFETCH_MAX, host, stream=side)
    side.synchronize()
    assert [(s, b) for s, b, _, _ in tail] == [(s, b) for s, b, _, _ in oracle_plan(rest, len(rest))]
    assert run.ctx.prefetch_plan(8) == []
    for sid in run.ids:
        assert run.ctx.export_records(sid).tobytes() == before[sid].tobytes()
        for b, p in enumerate(run.ctx.seq_info(sid)[3]):
            assert run.ctx.page_bytes_of(p).cpu().numpy().tobytes() == pages_before[(sid, b)]
    with pytest.raises(K.KvsError) as e:
        run.ctx.prefetch_plan(K.KVS_PREFETCH_MAX + 1)
    assert e.value.code == K.KVS_EINVAL
    for _ in range(2):
        run.compare(run.step(None))
    run.close()


def test_error_paths():
    # steps only sizes the table row (7 blocks) so the append below fails on
    # the pool (1 free page), not on the row length
    wl = W.workload("tiny", prefill_lens=(32,), pool_pages=3, steps=60)
    run = Run(wl, 0.1)
    ctx = run.ctx
    sid = run.ids[0]
    with pytest.raises(K.KvsError) as e:
        ctx.seq_add(sid)
    assert e.value.code == K.KVS_EEXIST
    Kt, Vt = W.kv_tokens(wl, 0, 32, 32 + 40, "cuda")
    with pytest.raises(K.KvsError) as e:           # needs 3 new pages, 1 free
        ctx.append_tokens(sid, Kt, Vt)
    assert e.value.code == K.KVS_ENOMEM
    Kt, Vt = W.kv_tokens(wl, 0, 32, 32 + 200, "cuda")
    with pytest.raises(K.KvsError) as e:           # would need 15 blocks in a 7-block row
        ctx.append_tokens(sid, Kt, Vt)
    assert e.value.code == K.KVS_EINVAL
    assert ctx.seq_info(sid)[1] == 32               # nothing appended
    with pytest.raises(K.KvsError) as e:
        ctx.decode_step([12345], torch.zeros((1, wl.L, wl.Hq, wl.d), dtype=torch.bfloat16,
                                             device="cuda"),
                        torch.zeros((1, wl.L, wl.Hq, wl.d), device="cuda"))
    assert e.value.code == K.KVS_ENOTFOUND
    with pytest.raises(K.KvsError) as e:
        ctx.readmit([(sid, 0)], _pinned(wl.page_bytes))
    assert e.value.code == K.KVS_EEXIST
    with pytest.raises(K.KvsError) as e:
        ctx.readmit([(sid, 7)], _pinned(wl.page_bytes))
    assert e.value.code == K.KVS_ENOTFOUND
    with pytest.raises(K.KvsError) as e:
        ctx.score_update()
    assert e.value.code == K.KVS_EINVAL
    # truncation: a host buffer of one page for a longer list
    q = W.queries(wl, 0, 1, "cuda").unsqueeze(0).contiguous()
    out = torch.empty((1, wl.L, wl.Hq, wl.d), device="cuda")
    ctx.decode_step([sid], q, out)
    ctx.debug_set_mass([sid], torch.zeros((1, run.mb), device="cuda"))
    ctx.debug_advance(100)
    ctx.debug_set_mass([sid], torch.zeros((1, run.mb), device="cuda"))
    ctx.score_update()
    rc, r = ctx.select_and_gather(K.KVS_SELECT_LOWFRAC, _pinned(wl.page_bytes), frac=1.0)
    assert rc == K.KVS_ETRUNC and r.n_pages == 2 and r.n_staged == 1
    ctx.check_device()
    run.close()


def test_mirror_mode_sends_each_full_page_once():
    wl = W.workload("tiny", prefill_lens=(100, 64), pool_pages=20, steps=5, skew=True)
    run = Run(wl, 0.15)
    mirror = _pinned(wl.pool_pages * wl.page_bytes)
    staged = []
    for _ in range(wl.steps):
        res = run.step(mirror, flags=K.KVS_GATHER_MIRROR)
        run.compare(res)
        staged.append(res["gather"].n_staged)
        pb = run.ctx.page_bytes
        hb = mirror.numpy()
        for (sid, b), slot in zip(res["ids"], res["slots"]):
            assert hb[slot * pb:(slot + 1) * pb].tobytes() == run.oracle_page(sid, b)
    assert staged[0] > 0 and max(staged[1:]) <= 2
    run.close()


# ------------------------------------------------- asynchronous mirror mode


def _counts(r):
    return (r.n_selected, r.n_pages, r.n_staged, r.n_demoted, r.bytes_to_host)


@pytest.mark.parametrize("name,kw", [
    ("tiny", dict(prefill_lens=(100, 64), pool_pages=20, steps=6, skew=True)),
    ("l70b_8k", dict(L=4, prefill_lens=(1000, 300, 17), pool_pages=100, steps=5))])
def test_async_mirror_matches_sync(name, kw):
    """KVS_GATHER_MIRROR | KVS_GATHER_ASYNC (stale pages written by a device
    kernel through the mirror's mapping, counts from kvs_gather_counts)
    against the synchronous mirror on a second context fed the same steps:
    same ids, slots and counts every step, byte-equal host mirrors, and the
    mirrored pages equal the oracle's page assembly."""
    wl = W.workload(name, **kw)
    sync_run, async_run = Run(wl, 0.15), Run(wl, 0.15, oracle_on=False)
    pb = sync_run.ctx.page_bytes
    m_sync, m_async = _pinned(wl.pool_pages * pb), _pinned(wl.pool_pages * pb)
    m_sync.zero_()
    m_async.zero_()      # pages neither context writes compare equal too
    staged = 0
    for _ in range(wl.steps):
        a = sync_run.step(m_sync, flags=K.KVS_GATHER_MIRROR)
        b = async_run.step(m_async, flags=K.KVS_GATHER_MIRROR | K.KVS_GATHER_ASYNC)
        sync_run.compare(a)
        assert a["ids"] == b["ids"] and a["slots"] == b["slots"]
        assert _counts(a["gather"]) == _counts(b["gather"])
        assert torch.equal(a["out"], b["out"])
        assert m_sync.numpy().tobytes() == m_async.numpy().tobytes()
        hb = m_async.numpy()
        for (sid, blk), slot in zip(b["ids"], b["slots"]):
            if slot >= 0:
                assert hb[slot * pb:(slot + 1) * pb].tobytes() == sync_run.oracle_page(sid, blk)
        staged += b["gather"].n_staged
    assert staged > 0
    async_run.ctx.check_device()
    sync_run.close()
    async_run.close()


def test_async_ids_only_in_2bit_context():
    """2-bit context: KVS_GATHER_ASYNC returns the same THRESH and LOWFRAC
    lists as the synchronous call, counts through kvs_gather_counts."""
    wl = W.workload("l70b_8k", L=2, prefill_lens=(300, 500), pool_pages=60, steps=3)
    run = Run(wl, 0.15, kv_dtype=K.KVS_KV_KIVI2, kivi_groups=32)
    for _ in range(wl.steps):
        run.compare(run.step(None))
    nrec = sum(len(run.ctx.export_records(s)) for s in run.ids)
    for mode, frac in ((K.KVS_SELECT_THRESH, 0.0), (K.KVS_SELECT_LOWFRAC, 0.25)):
        i1 = torch.zeros(2 * nrec, dtype=torch.int64, device="cuda")
        i2 = torch.zeros(2 * nrec, dtype=torch.int64, device="cuda")
        rc, r1 = run.ctx.select_and_gather(mode, frac=frac, ids=i1)
        rc2, r0 = run.ctx.select_and_gather(mode, frac=frac, flags=K.KVS_GATHER_ASYNC, ids=i2)
        assert rc == rc2 == K.KVS_OK and _counts(r0) == (0, 0, 0, 0, 0)
        r2 = run.ctx.gather_counts()
        torch.cuda.synchronize()
        assert _counts(r1) == _counts(r2) and r1.n_selected > 0
        n = r1.n_selected
        assert torch.equal(i1[:2 * n], i2[:2 * n])
    run.close()


def test_async_error_paths():
    wl = W.workload("tiny", prefill_lens=(100,), pool_pages=20, steps=1)
    run = Run(wl, 0.15, oracle_on=False)
    run.step(None)
    pb = run.ctx.page_bytes
    mirror = _pinned(wl.pool_pages * pb)
    with pytest.raises(K.KvsError) as e:        # no asynchronous select yet
        run.ctx.gather_counts()
    assert e.value.code == K.KVS_EINVAL
    for flags in (K.KVS_GATHER_ASYNC, K.KVS_GATHER_ASYNC | K.KVS_GATHER_DEMOTE, 64):
        with pytest.raises(K.KvsError) as e:
            run.ctx.select_and_gather(K.KVS_SELECT_THRESH, mirror, flags=flags)
        assert e.value.code == K.KVS_EINVAL
    # pageable host memory cannot take device writes: refused before any work
    page = np.zeros(wl.pool_pages * pb, dtype=np.uint8)
    a = K.kvs_gather_args()
    a.mode = K.KVS_SELECT_THRESH
    a.flags = K.KVS_GATHER_MIRROR | K.KVS_GATHER_ASYNC
    a.host_dst = page.ctypes.data
    a.host_dst_bytes = page.nbytes
    r = K.kvs_gather_result()
    rc = K.lib().kvs_select_and_gather(run.ctx.h, ctypes.byref(a), ctypes.byref(r))
    assert rc == K.KVS_EINVAL and b"page-locked" in K.lib().kvs_last_error(run.ctx.h)
    # a valid asynchronous call after the refusals
    rc, _ = run.ctx.select_and_gather(K.KVS_SELECT_THRESH, mirror,
                                      flags=K.KVS_GATHER_MIRROR | K.KVS_GATHER_ASYNC)
    assert rc == K.KVS_OK and run.ctx.gather_counts().n_selected >= 0
    run.ctx.check_device()
    run.close()


def test_async_steps_enqueued_back_to_back():
    """The pipelined use of KVS_GATHER_ASYNC: 24 steps (append, decode, score,
    asynchronous mirror select) enqueued with no host wait between them, the
    counts of each select read one step later; against a synchronising
    context fed the same inputs: every step's output, the final records and
    the host mirrors are bit-equal, and the staged-page totals agree."""
    wl = W.workload("l70b_8k", L=4, prefill_lens=(700, 300, 33), pool_pages=80, steps=24)
    sync_run, async_run = Run(wl, 0.15, oracle_on=False), Run(wl, 0.15, oracle_on=False)
    pb = sync_run.ctx.page_bytes
    m_sync, m_async = _pinned(wl.pool_pages * pb), _pinned(wl.pool_pages * pb)
    m_sync.zero_()
    m_async.zero_()
    ids = sync_run.ids
    ntok = list(wl.prefill_lens)
    rows, qs = [], []
    for t in range(1, wl.steps + 1):
        new = [W.kv_tokens(wl, s, ntok[s] + t - 1, ntok[s] + t, "cuda") for s in range(wl.nseq)]
        rows.append((torch.cat([k for k, _ in new]).contiguous(), torch.cat([v for _, v in new]).contiguous()))
        qs.append(torch.stack([W.queries(wl, s, t, "cuda") for s in range(wl.nseq)]).contiguous())
    torch.cuda.synchronize()
    shape = (wl.nseq, wl.L, wl.Hq, wl.d)
    outs_s = [torch.empty(shape, dtype=torch.float32, device="cuda") for _ in range(wl.steps)]
    outs_a = [torch.empty(shape, dtype=torch.float32, device="cuda") for _ in range(wl.steps)]
    side = torch.cuda.Stream()
    staged_s = staged_a = 0
    pending = False
    for t in range(wl.steps):
        a = async_run.ctx
        a.append_step(ids, *rows[t])
        a.decode_step(ids, qs[t], outs_a[t])
        a.score_update()
        if pending:                      # the previous step's counts, read one step late
            staged_a += a.gather_counts().n_staged
        rc, r0 = a.select_and_gather(K.KVS_SELECT_THRESH, m_async,
                                     flags=K.KVS_GATHER_MIRROR | K.KVS_GATHER_ASYNC)
        assert rc == K.KVS_OK and r0.n_selected == 0
        pending = True
        s = sync_run.ctx
        s.append_step(ids, *rows[t])
        s.decode_step(ids, qs[t], outs_s[t])
        s.score_update()
        rc, r = s.select_and_gather(K.KVS_SELECT_THRESH, m_sync, flags=K.KVS_GATHER_MIRROR,
                                    side_stream=side)
        staged_s += r.n_staged
    staged_a += async_run.ctx.gather_counts().n_staged
    side.synchronize()
    torch.cuda.synchronize()
    for t in range(wl.steps):
        assert torch.equal(outs_s[t], outs_a[t]), t
    for sid in ids:
        assert sync_run.ctx.export_records(sid).tobytes() == async_run.ctx.export_records(sid).tobytes()
    assert m_sync.numpy().tobytes() == m_async.numpy().tobytes()
    assert staged_a == staged_s > 0
    async_run.ctx.check_device()
    sync_run.close()
    async_run.close()
