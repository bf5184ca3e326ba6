"""Failure paths without a GPU fault: failures are made on the host (an
injected failing allocation, host waits that never see completion) or caught
by the kernels' own bounds checks (an out-of-range block-table entry, which
the decode kernel records and replaces by a valid page before any access)."""
import pytest
import torch

import paged_kv_cache_flash_gb300 as K
import workloads as W
from gpu_harness import Run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_flash_gb300 import build
    build.build()
    yield
    K.debug_inject(0, 0)


def test_injected_pinned_allocation_failure_leaves_nothing_behind():
    cfg = K.make_config(2, 8, 2, 64, 17, 1, 18)
    K.debug_inject(K.KVS_FAULT_HOSTALLOC)
    with pytest.raises(K.KvsError) as e:
        K.Context(cfg)
    assert e.value.code == K.KVS_ENOMEM and "injected" in str(e.value)
    ctx = K.Context(cfg)                        # one shot: the next create works
    ctx.check_device()
    ctx.close()


def test_host_waits_time_out_and_recover():
    wl = W.workload("tiny", prefill_lens=(100,), pool_pages=20, steps=2)
    run = Run(wl, 0.15)
    run.compare(run.step(None))
    K.debug_inject(K.KVS_FAULT_WAIT, 30)
    try:
        with pytest.raises(K.KvsError) as e:
            run.ctx.check_device()
        assert e.value.code == K.KVS_ETIMEOUT
        with pytest.raises(K.KvsError) as e:      # the selection's read-back
            run.ctx.select_and_gather(K.KVS_SELECT_THRESH)
        assert e.value.code == K.KVS_ETIMEOUT
    finally:
        K.debug_inject(0, 0)
    torch.cuda.synchronize()
    run.ctx.check_device()
    run.compare(run.step(None))                   # the context stays usable
    run.close()


def test_out_of_range_table_entry_is_caught_by_the_decode_kernel():
    wl = W.workload("tiny", prefill_lens=(100,), pool_pages=20, steps=1)
    run = Run(wl, 0.15, oracle_on=False)
    sid = run.ids[0]
    slot = run.ctx.seq_info(sid)[0]
    table = run.ctx.table.view(torch.int32)[: wl.nseq * run.mb].view(wl.nseq, run.mb)
    good = int(table[slot, 3].item())
    table[slot, 3] = wl.pool_pages + 1000       # out of range on the device only
    q = torch.zeros((1, wl.L, wl.Hq, wl.d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((1, wl.L, wl.Hq, wl.d), device="cuda")
    run.ctx.decode_step([sid], q, out)
    with pytest.raises(K.KvsError) as e:
        run.ctx.check_device()
    assert e.value.code == K.KVS_EDEVICE and "bad page 1" in str(e.value)
    table[slot, 3] = good
    run.ctx.decode_step([sid], q, out)
    run.ctx.check_device()                      # the word was cleared; decode is clean again
    run.close()
