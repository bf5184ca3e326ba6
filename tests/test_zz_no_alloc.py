"""The allocation-free decode entry point (kvs_decode_noalloc), through the
C ABI, against the fp64 oracle and against the regular entry point
(kvs_decode_step).

kvs_decode_noalloc serves callers that are handed only their input and
output buffers and may not allocate device memory themselves (a plugin or
custom operator living inside another framework's memory budget, or a
serving loop that allows no allocation after start-up).  Its scratch is a
fixed array inside the library, shared by every call, so two calls in a row
must each give the right result, whatever the previous call left behind:
a call repeated after another one must give the same bits.  Against the
oracle the bar is the path's stated tolerances.  Against kvs_decode_step,
which runs the same kernels over another split of the blocks into chunks:
the block masses within a few fp32 rounding steps, the outputs within the
rounding of the softmax weights to bf16 before the P.V product (each path
rounds them relative to its own chunk's running maximum).  This file is
collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import paged_kv_cache_flash_gb300 as K
import workloads as W

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2          # against the oracle: attention output, max abs
MASS_TOL = 1e-4         # against the oracle: block mass, abs
SAME_MASS_TOL = 1e-6    # against kvs_decode_step: same kernels, other chunking


def same_out_tol(V):
    """Bound on |out - out'| between two chunkings: each path's weights are
    rounded to bf16 (relative error <= 2^-9) before the P.V product, so each
    output lies within 2^-9 max|v| of the unrounded weighted mean, the two
    within twice that; plus fp32 accumulation slack."""
    return 2.0 ** -8 * float(V.float().abs().max()) + 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_flash_gb300 import build
    build.build()


def _noalloc(ctx, wl, sid, q, out, mass, status, msg, table=None):
    slot, ntok, nb, _ = ctx.seq_info(sid)
    mb = ctx.cfg.max_blocks_per_seq
    if table is None:
        table = ctx.table.data_ptr() + slot * mb * 4
    return K.lib().kvs_decode_noalloc(wl.L, wl.Hq, wl.Hkv, wl.d, ctx.pool.data_ptr(),
                                      ctx.cfg.pool_blocks, table, ntok, q.data_ptr(),
                                      out.data_ptr(), mass.data_ptr(),
                                      None if status is None else status.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream, msg, len(msg))


def _two_calls_in_a_row(wl, ids, pool_pages, max_blocks):
    """Prefill every sequence, then for each in turn: kvs_decode_step, then
    kvs_decode_noalloc over the same pages and query; both against the fp64
    oracle, and against each other."""
    cfg = K.make_config(wl.L, wl.Hq, wl.Hkv, wl.d, pool_pages, len(ids), max_blocks,
                        pool_seed=wl.seed)
    ctx = K.Context(cfg)
    kv = []
    for s, sid in enumerate(ids):
        ctx.seq_add(sid)
        Kt, Vt = W.kv_tokens(wl, s, 0, wl.prefill_lens[s], "cuda")
        ctx.append_tokens(sid, Kt, Vt)
        kv.append((Kt.cpu(), Vt.cpu()))
        del Kt, Vt
    msg = ctypes.create_string_buffer(256)
    status = torch.full((2,), 0xFFFF, dtype=torch.int32, device="cuda")
    errs = []
    first = None
    for s, sid in enumerate(ids):
        q = W.queries(wl, s, 1, "cuda").unsqueeze(0).contiguous()
        ref = torch.empty((1, wl.L, wl.Hq, wl.d), dtype=torch.float32, device="cuda")
        ctx.decode_step([sid], q, ref)
        slot, _, nb, _ = ctx.seq_info(sid)
        ref_mass = ctx.mass()[slot, :nb].clone()
        out = torch.full_like(ref, float("nan"))
        mass = torch.full((nb,), float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc(ctx, wl, sid, q, out, mass, status, msg)
        assert rc == K.KVS_OK, msg.value
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0]
        assert torch.isfinite(out).all() and torch.isfinite(mass).all()
        e_out = (out - ref).abs().max().item()
        e_mass = (mass - ref_mass).abs().max().item()
        assert e_out <= same_out_tol(kv[s][1]) and e_mass <= SAME_MASS_TOL, (e_out, e_mass)
        if first is None:
            first = (sid, q, out.clone(), mass.clone())
        orc = O.decode_with_mass(q[0].cpu(), kv[s][0], kv[s][1], L=wl.L, Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d)
        o_out = float(np.abs(out[0].cpu().numpy() - orc["out"]).max())
        o_mass = float(np.abs(mass.cpu().numpy().astype(np.float64) - orc["mass"]).max())
        assert o_out <= OUT_TOL and o_mass <= MASS_TOL, (o_out, o_mass)
        errs.append((e_out, e_mass, o_out, o_mass))
    # the first call again, after the other one filled the scratch: same bits
    sid, q, out0, mass0 = first
    out = torch.full_like(out0, float("nan"))
    mass = torch.full_like(mass0, float("nan"))
    assert _noalloc(ctx, wl, sid, q, out, mass, status, msg) == K.KVS_OK, msg.value
    torch.cuda.synchronize()
    assert torch.equal(out, out0) and torch.equal(mass, mass0) and status.tolist() == [0, 0]
    ctx.check_device()
    ctx.close()
    return errs


def test_noalloc_70b_shape_two_calls_in_a_row():
    # 80-layer 70B shape (4 KV heads per warp group); a longer sequence first
    # (188 blocks: two 64-block chunks and a short one), then a shorter one
    # (63 blocks: one short chunk), so the second call runs over scratch the
    # first one filled
    wl = W.workload("l70b_8k", prefill_lens=(3001, 1000), pool_pages=260, steps=0)
    print("70b", _two_calls_in_a_row(wl, [11, 7], 260, 200))


def test_noalloc_small_geometry_two_calls_in_a_row():
    # d = 64, 4:1 groups over 2 KV heads (2 KV heads per warp group):
    # 69 blocks (a full chunk and a 5-block one), then a one-token sequence
    wl = W.workload("tiny", prefill_lens=(1100, 1), pool_pages=80, steps=0, skew=True)
    print("small", _two_calls_in_a_row(wl, [3, 4], 80, 80))


def test_noalloc_reports_a_bad_table_entry():
    """A block-table entry outside the pool (here a demoted entry, -1, and
    one past the end): the kernel reads page 0 in its place, and status
    reports it with the offending value; a good call after it reports
    nothing."""
    wl = W.workload("tiny", prefill_lens=(100,), pool_pages=12, steps=0)
    cfg = K.make_config(wl.L, wl.Hq, wl.Hkv, wl.d, 12, 1, 16, pool_seed=1)
    ctx = K.Context(cfg)
    ctx.seq_add(3)
    Kt, Vt = W.kv_tokens(wl, 0, 0, 100, "cuda")
    ctx.append_tokens(3, Kt, Vt)
    q = W.queries(wl, 0, 1, "cuda").contiguous()
    _, _, nb, table = ctx.seq_info(3)
    out = torch.empty((wl.L, wl.Hq, wl.d), dtype=torch.float32, device="cuda")
    mass = torch.empty(nb, dtype=torch.float32, device="cuda")
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    msg = ctypes.create_string_buffer(256)
    for bad in (-1, 12):
        t = torch.tensor(table, dtype=torch.int32, device="cuda")
        t[3] = bad
        rc = _noalloc(ctx, wl, 3, q, out, mass, status, msg, table=t.data_ptr())
        assert rc == K.KVS_OK, msg.value
        torch.cuda.synchronize()
        err, info = (x & 0xFFFFFFFF for x in status.tolist())
        assert err & 1 and info == (bad & 0xFFFFFFFF) | 0x80000000, (err, info)
    rc = _noalloc(ctx, wl, 3, q, out, mass, status, msg)
    assert rc == K.KVS_OK
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0]
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
                                    12289, q.data_ptr(), out.data_ptr(), mass.data_ptr(), None,
                                    torch.cuda.current_stream().cuda_stream, msg, len(msg))
    assert rc == K.KVS_EINVAL
    assert b"maximum" in msg.value
    ctx.close()
