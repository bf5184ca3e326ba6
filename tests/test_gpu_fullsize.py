"""Full-size parity of the CUDA path with the fp64 oracle on the batched,
128K and mixed-eviction workloads (the launch configuration bench.py times).
Each sequence's attention, mass and records depend on it alone, so the
oracle follows a subset of sequences where the full set would not fit the
host's memory or time; the global selections are checked by properties."""
import numpy as np
import pytest
import torch

import oracle as O
import paged_kv_cache_flash_gb300 as K
import workloads as W
from gpu_harness import Run
from test_gpu_parity import _check_gather, _pinned

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_flash_gb300 import build
    build.build()


def test_batch16_shared_prefix_full_size():
    """16 sequences of 1,024..8,192 tokens sharing a 64-block prefix
    (refcount 16), every sequence followed by the oracle, 2 steps."""
    wl = W.workload("l70b_batch16", steps=2)
    run = Run(wl, 0.15)
    host = _pinned(wl.pool_pages * wl.page_bytes)
    for _ in range(wl.steps):
        res = run.step(host)
        summ = run.compare(res)
        _check_gather(run, res, host, sample=48)
        # the shared prefix pages are gathered only when all 16 users list them
        pre = {b for b in range(64)}
        listed = {}
        for (sid, b) in res["ids"]:
            if b in pre:
                listed.setdefault(b, set()).add(sid)
        for b, users in listed.items():
            slots = [sl for (sid, bb), sl in zip(res["ids"], res["slots"]) if bb == b]
            if len(users) < wl.nseq:
                assert all(sl == -1 for sl in slots)
            else:
                assert len(set(slots)) == 1 and slots[0] >= 0
    print("batch16", summ)
    run.close()


def test_fp8_8k_full_size():
    """The 8K workload with FP8 E4M3 pages (scales 1.0), 2 steps, full oracle."""
    wl = W.workload("l70b_8k", steps=2)
    run = Run(wl, 0.15, kv_dtype=K.KVS_KV_FP8_E4M3)
    host = _pinned(wl.pool_pages * run.ctx.page_bytes)
    for _ in range(wl.steps):
        res = run.step(host)
        summ = run.compare(res)
        _check_gather(run, res, host, sample=32)
    print("fp8 8k", summ)
    run.close()


def test_kivi_8k_full_size():
    """The 8K workload with 2-bit groups behind the residual window, 2 steps,
    full oracle on the effective values; 3 group pages byte for byte."""
    from test_gpu_parity import _check_kivi_groups
    wl = W.workload("l70b_8k", steps=2)
    run = Run(wl, 0.15, kv_dtype=K.KVS_KV_KIVI2, kivi_groups=8192 // 32 + 4)
    for _ in range(wl.steps):
        summ = run.compare(run.step(None))
    assert _check_kivi_groups(run, sample=3) == O.kivi_quantized_tokens(8194) // 32
    print("kivi 8k", summ)
    run.close()


def test_128k_full_size():
    """1 sequence of 131,072 tokens (8,192 blocks, 40 GiB), 2 steps: outputs,
    masses and records against the full oracle; the P < 0.3 list in full and
    the first 64 gathered pages byte for byte (host buffer of 64 pages)."""
    wl = W.workload("l70b_128k", steps=2)
    run = Run(wl, 0.05)
    host = _pinned(64 * wl.page_bytes)
    for _ in range(wl.steps):
        res = run.step(host)
        assert res["rc"] == K.KVS_ETRUNC and res["gather"].n_staged == 64
        summ = run.compare(res)
        _check_gather(run, res, host, sample=64, limit=64)
    print("128k", summ)
    run.close()


def test_mixed32_demote_readmit_full_size():
    """32 sequences of 4,096..16,384 tokens (~104 GiB) in a pool sized to
    110 % of need, alpha 0.05: 8 steps (oracle following 3 sequences), the
    10 % lowest-P blocks demoted to pinned host and re-admitted, 2 more steps."""
    wl = W.workload("l70b_mixed32", steps=10)
    follow = [0, 13, 31]
    run = Run(wl, 0.05, oracle_seqs=follow)
    for _ in range(8):
        run.compare(run.step(None))
    before = {sid: run.ctx.export_records(sid) for sid in run.ids}
    allrec = np.concatenate([before[s] for s in sorted(before)])
    nrec = len(allrec)
    k = O.lowfrac_k(nrec, 0.10)
    host = _pinned(k * wl.page_bytes)
    ids = torch.zeros(2 * nrec, dtype=torch.int64, device="cuda")
    # checksums of every page before demotion (device-side, round-trip check)
    sums_before = {}
    for sid in run.ids:
        for b, p in enumerate(run.ctx.seq_info(sid)[3]):
            sums_before[(sid, b)] = int(run.ctx.page_bytes_of(p).view(torch.int64).sum().item())
    free0 = run.ctx.free_pages()
    rc, r = run.ctx.select_and_gather(K.KVS_SELECT_LOWFRAC, host, frac=0.10,
                                      flags=K.KVS_GATHER_DEMOTE, ids=ids)
    torch.cuda.synchronize()
    assert rc == K.KVS_OK and r.n_selected == k == r.n_demoted
    assert run.ctx.free_pages() == free0 + k
    got = [tuple(x) for x in ids.view(-1, 2)[:k].cpu().tolist()]
    assert got == sorted(got)
    # property of the k smallest (P, record order): every chosen record beats every other
    order = {(int(a), int(b)): i for i, (a, b) in enumerate(zip(allrec["seq_id"], allrec["block_idx"]))}
    prio = {key: float(allrec["prio"][i]) for key, i in order.items()}
    chosen = set(got)
    worst_in = max((prio[x], order[x]) for x in chosen)
    best_out = min((prio[x], order[x]) for x in order if x not in chosen)
    assert worst_in < best_out
    # demoted pages of followed sequences equal the oracle's page assembly
    hb = host.numpy()
    pb = wl.page_bytes
    checked = 0
    for i, (sid, b) in enumerate(got):
        if sid in run.orc and checked < 24:
            assert hb[i * pb:(i + 1) * pb].tobytes() == run.oracle_page(sid, b)
            checked += 1
    run.ctx.readmit(got, host)
    torch.cuda.synchronize()
    for sid in run.ids:
        assert run.ctx.export_records(sid).tobytes() == before[sid].tobytes()
    for (sid, b) in got:
        p = run.ctx.seq_info(sid)[3][b]
        assert int(run.ctx.page_bytes_of(p).view(torch.int64).sum().item()) == sums_before[(sid, b)]
    for _ in range(2):
        run.compare(run.step(None))
    run.ctx.check_device()
    run.close()
