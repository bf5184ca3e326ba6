"""The allocation-free decode entry point (kvs_decode_noalloc) against the
regular one (kvs_decode_step), through the C ABI.

kvs_decode_noalloc serves callers that are handed only their input and
output buffers and may not allocate device memory themselves (a plugin or
custom operator living inside another framework's memory budget, or a
serving loop that allows no allocation after start-up).  Its scratch is a
fixed array inside the library, shared by every call, so two calls in a row
must each give the same result as the regular path, whatever the previous
call left behind.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_flash_gb300 as K
import workloads as W

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
MASS_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_flash_gb300 import build
    build.build()


def _noalloc(ctx, wl, sid, q, out, mass, msg):
    slot, ntok, nb, _ = ctx.seq_info(sid)
    mb = ctx.cfg.max_blocks_per_seq
    table = ctx.table.data_ptr() + slot * mb * 4
    return K.lib().kvs_decode_noalloc(wl.L, wl.Hq, wl.Hkv, wl.d, ctx.pool.data_ptr(),
                                      ctx.cfg.pool_blocks, table, ntok, q.data_ptr(),
                                      out.data_ptr(), mass.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream, msg, len(msg))


def test_noalloc_matches_decode_step_two_calls_in_a_row():
    # 80-layer 70B shape; a longer sequence first, then a shorter one, so the
    # second call runs over scratch the first one filled
    wl = W.workload("l70b_8k", prefill_lens=(3001, 1000), pool_pages=260, steps=0)
    cfg = K.make_config(wl.L, wl.Hq, wl.Hkv, wl.d, wl.pool_pages, wl.nseq, 200,
                        pool_seed=wl.seed)
    ctx = K.Context(cfg)
    ids = [11, 7]
    for s, sid in enumerate(ids):
        ctx.seq_add(sid)
        Kt, Vt = W.kv_tokens(wl, s, 0, wl.prefill_lens[s], "cuda")
        ctx.append_tokens(sid, Kt, Vt)
    msg = ctypes.create_string_buffer(256)
    for s, sid in enumerate(ids):
        q = W.queries(wl, s, 1, "cuda").unsqueeze(0).contiguous()
        ref = torch.empty((1, wl.L, wl.Hq, wl.d), dtype=torch.float32, device="cuda")
        ctx.decode_step([sid], q, ref)
        slot, _, nb, _ = ctx.seq_info(sid)
        ref_mass = ctx.mass()[slot, :nb].clone()
        out = torch.full_like(ref, float("nan"))
        mass = torch.full((nb,), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc(ctx, wl, sid, q, out, mass, msg)
        assert rc == K.KVS_OK, msg.value
        torch.cuda.synchronize()
        assert torch.isfinite(out).all() and torch.isfinite(mass).all()
        assert (out - ref).abs().max().item() <= OUT_TOL
        assert (mass - ref_mass).abs().max().item() <= MASS_TOL
        assert abs(mass.double().sum().item() - 1.0) < 1e-4
    ctx.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    wl = W.workload("l70b_8k", prefill_lens=(16,), pool_pages=4, steps=0)
    cfg = K.make_config(wl.L, wl.Hq, wl.Hkv, wl.d, wl.pool_pages, 1, 1000, pool_seed=1)
    ctx = K.Context(cfg)
    ctx.seq_add(3)
    Kt, Vt = W.kv_tokens(wl, 0, 0, 16, "cuda")
    ctx.append_tokens(3, Kt, Vt)
    q = W.queries(wl, 0, 1, "cuda").contiguous()
    out = torch.empty((wl.L, wl.Hq, wl.d), dtype=torch.float32, device="cuda")
    mass = torch.empty(1000, dtype=torch.float32, device="cuda")
    msg = ctypes.create_string_buffer(256)
    slot = ctx.seq_info(3)[0]
    table = ctx.table.data_ptr() + slot * 1000 * 4
    rc = K.lib().kvs_decode_noalloc(wl.L, wl.Hq, wl.Hkv, wl.d, ctx.pool.data_ptr(), 4, table,
                                    12289, q.data_ptr(), out.data_ptr(), mass.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream, msg, len(msg))
    assert rc == K.KVS_EINVAL
    assert b"maximum" in msg.value
    ctx.close()
