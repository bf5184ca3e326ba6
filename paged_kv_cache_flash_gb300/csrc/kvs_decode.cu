// Paged GQA decode with per-block attention mass (sm_103a).
//
// Sources: "KV-Cache Offloading for LLM Inference -- Visual Reference" s.4
// (a decode step reads every cached token of the sequence) and the "GQA
// per-head attention as scoring streams" page (query heads grouped 8:1 onto
// a KV head; every (layer, KV head) stream contributes to one mass per
// (sequence, 16-token block)).
//
// Structure of one step:
//   decode_kernel  -- persistent grid of independent warps.  Each warp claims
//                     work items (sequence, layer, KV head, chunk: 128-block
//                     chunks first, 16-block chunks over the end of each
//                     stream, claimed chunk by chunk) from a global counter,
//                     each shortly before its ring needs the item's first
//                     block, and keeps its own TMA ring of the head's K and V
//                     sub-pages streaming across item boundaries (128-byte
//                     swizzle, bounded mbarrier waits).  Warp-level
//                     tensor-core MMAs compute
//                       S^T[16 tokens][8 heads] = K . Q^T
//                       O^T[d][8 heads]        += V^T . P^T
//                     with an online softmax in registers.  Per block it writes
//                     the block's log2-sum-exp for each query head; per item
//                     the running max, sum and unnormalised output.
//                     bf16 pages: bf16 MMAs, 3-stage rings, 8 warps per SM.
//                     FP8 E4M3 pages ("Fitting a Million Tokens", s.02): S by
//                     e4m3 MMAs over the stored codes with Q as two exact
//                     E4M3 terms, O by f16 MMAs over codes converted in
//                     registers; 4-stage rings, 12 warps per SM.
//                     (2-bit KIVI group pages are decoded by kvs_kivi.cu; the
//                     page items of such a sequence cover its residual blocks.)
//   combine_kernel -- merges a stream's chunks: per head log2-sum-exp LSE_h,
//                     the normalised output and the stream's block masses
//                     (kvs_combine.cu).
//   mass_kernel    -- M(b) = 1/(L*Hq) * sum_{l,h} 2^(lse_blk(l,h,b) - LSE_h),
//                     summed in a fixed order (deterministic); scores the
//                     records when asked.
#include <cuda_bf16.h>

#include "kvs_internal.h"
#include "kvs_pdl.cuh"
#include "kvs_ptx.h"

namespace kvs {
namespace {

using namespace ptx;

struct DecodeArgs {
    Geo g;
    Work w;
    const uint16_t *q;
    const int32_t *table;
    uint32_t n_items;
    uint32_t wg;
};

// Bytes of one block's K and V sub-pages for one KV head.  bf16: boxes of
// [K,V][16 tok][64 dims]; FP8 codes: one box of [K,V][16 tok][128 dims].
constexpr uint32_t kClaimLead = 4;   // blocks between claiming an item and needing its pages

template <int D, bool FP8>
struct Tile {
    static constexpr int kHalf = FP8 ? 1 : D / 64;       // TMA boxes per stage
    static constexpr int kBoxBytes = 2 * 16 * 64 * 2;    // 4 KiB either way
    static constexpr int kStageBytes = kHalf * kBoxBytes;
    static constexpr int kBoxElems = FP8 ? 128 : 64;     // box width in elements
    // Shallow rings so that several CTAs of 4 warps share an SM (the same
    // bytes in flight per SM): a lone warp per SM sub-partition streams only
    // as fast as its own instruction latencies allow, so two or three warps
    // per sub-partition keep HBM busy when some have run out of items.
    // bf16: two CTAs, 3 x 8 KiB per warp; FP8: three CTAs, 4 x 4 KiB.
    static constexpr int kRing = FP8 ? 4 : 3;
    static constexpr int kMinCtas = FP8 ? 3 : 2;
    static constexpr int kWarpBytes = kRing * kStageBytes;
};

// Head dimension of row r (0..15) of O^T m-tile mt.  bf16: 16 mt + r.  FP8:
// m-tiles come in pairs (even, odd dims) per 32-dim group, from the V
// fragment load below: rows 0..7 -> dims 2r, rows 8..15 -> 16 + 2(r-8).
template <bool FP8>
__device__ __forceinline__ uint32_t o_dim(uint32_t mt, uint32_t r)
{
    if constexpr (FP8)
        return 32 * (mt >> 1) + (r < 8 ? 2 * r : 16 + 2 * (r - 8)) + (mt & 1);
    else
        return 16 * mt + r;
}

// A warp's TMA ring: blocks in flight, the stage the next issue fills, the
// stage the consumer waits on and that stage's mbarrier phase.
struct Ring {
    uint32_t inflight;
    uint32_t st_issue;
    uint32_t st_cons;
    uint32_t ph_cons;
};

// A claimed work item: one chunk of blocks of one (sequence, layer, KV head)
// stream, decoded by one warp.
struct Item {
    uint32_t valid;
    uint32_t ci;        // sequence (call order)
    uint32_t l;         // layer
    uint32_t kvh;       // KV head
    uint32_t b0;        // first block
    uint32_t nblk;      // blocks in the chunk
    uint32_t ntok;      // tokens of the sequence
    uint32_t part;      // partial index
    uint32_t lse0;      // blk_off + b0: column of the chunk's first block in lse_blk
};

// An item with its page ids: lane j holds those of blocks j, j+32, j+64, j+96.
struct Prep {
    Item it;
    int32_t pg[kMaxChunk / 32];
};

__device__ __forceinline__ Prep prepare_item(const DecodeArgs &a, uint32_t id, uint32_t lane)
{
    Prep p;
    p.it.valid = 0;
    p.it.nblk = 0;
    if (id >= a.n_items)
        return p;
    const DSet *ds = a.w.dset;
    const Geo &g = a.g;
    const uint32_t ci = find_seq(&ds->seq[0].item_off, sizeof(DSeq) / 4, ds->nseq, id);
    const DSeq &sq = ds->seq[ci];
    // KV head fastest: warps that claim consecutive items read adjacent
    // sub-pages of the same pages at about the same time (DRAM locality);
    // then layer, then chunk
    // (KIVI: the page items cover the blocks after the qb quantised ones,
    // and their partials follow the nchunk_q group-page chunks)
    // chunk-major: every stream's chunk c before any stream's chunk c + 1, so
    // the small last chunks are claimed last
    uint32_t local = id - sq.item_off;
    const uint32_t kvh = local % g.Hkv;
    local /= g.Hkv;
    const uint32_t l = local % g.L;
    const uint32_t chunk = local / g.L;
    const uint32_t r0 = chunk < sq.nbig ? chunk * ds->chunk_big
                                        : sq.nbig * ds->chunk_big + (chunk - sq.nbig) * ds->chunk_small;
    const uint32_t size = chunk < sq.nbig ? ds->chunk_big : ds->chunk_small;
    const uint32_t b0 = sq.qb + r0;
    const uint32_t nblk = min(size, sq.nb - b0);
    p.it.valid = 1;
    p.it.ci = ci;
    p.it.l = l;
    p.it.kvh = kvh;
    p.it.b0 = b0;
    p.it.nblk = nblk;
    p.it.ntok = sq.ntok;
    p.it.part = sq.part_off + (l * g.Hkv + kvh) * sq.nchunk + sq.nchunk_q + chunk;
    p.it.lse0 = sq.blk_off + b0;
    const int32_t *trow = a.table + static_cast<size_t>(sq.slot) * g.mb + b0;
#pragma unroll
    for (int q = 0; q < static_cast<int>(kMaxChunk / 32); ++q) {
        const uint32_t j = lane + 32 * q;
        int32_t pgid = j < nblk ? __ldg(trow + j) : 0;
        if (pgid < 0 || pgid >= static_cast<int32_t>(g.pool_blocks)) {
            atomicOr(a.w.err, kErrBadPage);
            atomicCAS(a.w.err_info, 0u, static_cast<uint32_t>(pgid) | 0x80000000u);
            pgid = 0;
        }
        p.pg[q] = pgid;
    }
    return p;
}

__device__ __forceinline__ int32_t page_of(const Prep &p, uint32_t j)
{
    // a select chain, not an indexed load: the page ids stay in registers
    static_assert(kMaxChunk == 32 || kMaxChunk == 64 || kMaxChunk == 128, "chunk cap");
    const uint32_t q = j >> 5;
    int32_t page = p.pg[0];
    if constexpr (kMaxChunk >= 64)
        page = q == 1 ? p.pg[1] : page;
    if constexpr (kMaxChunk >= 128)
        page = q == 2 ? p.pg[2] : (q == 3 ? p.pg[3] : page);
    return __shfl_sync(0xffffffffu, page, j & 31);
}

// Issues the next block of a warp's stream (items cur, then nxt) into its TMA
// ring; false when the stream position is not known yet.  Warp-uniform.
template <int D, bool FP8>
__device__ __forceinline__ bool issue_next(const CUtensorMap *tmap, const Geo &g, const Prep &cur,
                                           const Prep &nxt, bool have_nxt, bool &c_in_nxt,
                                           uint32_t &c_blk, Ring &rg, uint32_t ring_u32,
                                           uint64_t *bars, uint32_t lane)
{
    using T = Tile<D, FP8>;
    if (!c_in_nxt && c_blk >= cur.it.nblk) {
        if (!have_nxt || !nxt.it.valid)
            return false;
        c_in_nxt = true;
        c_blk = 0;
    }
    if (c_in_nxt && c_blk >= nxt.it.nblk)
        return false;
    const uint32_t l = c_in_nxt ? nxt.it.l : cur.it.l;
    const uint32_t kv = c_in_nxt ? nxt.it.kvh : cur.it.kvh;
    const int32_t page = c_in_nxt ? page_of(nxt, c_blk) : page_of(cur, c_blk);
    if (lane == 0) {
        const uint32_t st = rg.st_issue;
        const uint32_t bar = smem_u32(&bars[st]);
        mbar_expect_tx(bar, T::kStageBytes);
        const int c4 = page * static_cast<int>(g.L) + static_cast<int>(l);
        const uint64_t pol = l2_evict_first();      // pages are read once per step
#pragma unroll
        for (int h = 0; h < T::kHalf; ++h)
            tma_load_5d(ring_u32 + st * T::kStageBytes + h * T::kBoxBytes, tmap, bar,
                        h * T::kBoxElems, 0, static_cast<int>(kv), 0, c4, pol);
    }
    ++c_blk;
    ++rg.inflight;
    rg.st_issue = rg.st_issue + 1 == T::kRing ? 0 : rg.st_issue + 1;
    return true;
}

// Persistent kernel of fully independent warps.  Each warp claims work items
// (one KV-head stream chunk each) from a global counter, prepares the next
// one while it computes the last blocks of the current one, and keeps its own
// TMA ring of T::kRing blocks in flight across item boundaries.  No CTA-wide
// barrier.
template <int D, bool FP8>
__global__ void __launch_bounds__(128, Tile<D, FP8>::kMinCtas)
    decode_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeArgs a)
{
    using T = Tile<D, FP8>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[8][kStages];

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring_u32 = smem_u32(smem + warp * T::kWarpBytes);
    if (lane == 0) {
        for (int s = 0; s < T::kRing; ++s)
            mbar_init(smem_u32(&bars[warp][s]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
    // launched as a programmatic dependent of the decode-set upload: the CTAs
    // are placed while it runs, and nothing in global memory is touched
    // before it has completed.  Then the combine kernel (the next dependent)
    // may place its CTAs beside this persistent grid: they wait for its
    // completion, and start at once when it completes
    pdl_wait();
    pdl_trigger();

    const Geo &g = a.g;
    const uint32_t G = g.G;
    const uint32_t gq = lane >> 2;          // row group id in MMA fragments
    const uint32_t tq = lane & 3;           // thread in group
    const uint32_t h0 = 2 * tq, h1 = 2 * tq + 1;   // heads of this lane's S/O columns
    const float scale_log2 = rsqrtf(static_cast<float>(D)) * kLog2e * g.k_scale;
    const uint32_t nb_total = a.w.dset->nb_total;
    const uint32_t jm = lane >> 3, i8 = lane & 7;

    // bf16 query fragments (B operand of S^T = K Q^T) of head gq of an item:
    // loaded when the item is prepared, before the current item ends, so
    // that no item starts with a wait on them
    auto load_q = [&](const Item &itm, uint32_t (&dst)[D / 16][2]) {
        const bool valid = itm.valid && gq < G;
        const uint16_t *qh = a.q + ((static_cast<size_t>(valid ? itm.ci : 0) * g.L + (valid ? itm.l : 0)) * g.Hq +
                                    (valid ? itm.kvh * G + gq : 0)) * D;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            dst[ks][0] = valid ? __ldg(reinterpret_cast<const uint32_t *>(qh + ks * 16 + 2 * tq)) : 0u;
            dst[ks][1] = valid ? __ldg(reinterpret_cast<const uint32_t *>(qh + ks * 16 + 8 + 2 * tq)) : 0u;
        }
    };
    uint32_t qc[D / 16][2], qn[D / 16][2];   // bf16: current and next item

    // items are claimed one at a time, each shortly before the ring needs its
    // first block (kClaimLead blocks of compute hide the claim and the page-id
    // loads), so that a warp never holds work it has not nearly reached
    auto claim = [&]() -> uint32_t {
        uint32_t id = 0;
        if (lane == 0)
            id = atomicAdd(a.w.counter, 1u);
        return __shfl_sync(0xffffffffu, id, 0);
    };
    Prep cur = prepare_item(a, claim(), lane);
    if constexpr (!FP8)
        load_q(cur.it, qc);
    Prep nxt;
    nxt.it.valid = 0;
    nxt.it.nblk = 0;
    bool have_nxt = false;

    Ring rg{0, 0, 0, 0};
    bool c_in_nxt = false;                  // issue cursor: item (cur / nxt) and block
    uint32_t c_blk = 0;
    if (cur.it.valid)
        while (rg.inflight < T::kRing && issue_next<D, FP8>(&tmap, g, cur, nxt, have_nxt, c_in_nxt, c_blk, rg, ring_u32, bars[warp], lane)) {
        }

    while (cur.it.valid) {
        const Item it = cur.it;
        const uint32_t kvh = it.kvh;
        const uint32_t claim_at = it.nblk > T::kRing + kClaimLead ? it.nblk - T::kRing - kClaimLead : 0;

        // query fragments (B operand of S^T = K Q^T), head gq, and the scale
        // of the logits of this lane's heads h0, h1 (log2 domain)
        uint32_t qf[D / 16][2];
        float sl0 = scale_log2, sl1 = scale_log2;
        {
            const bool valid = gq < G;
            const uint16_t *qh = a.q + ((static_cast<size_t>(it.ci) * g.L + it.l) * g.Hq + kvh * G +
                                        (valid ? gq : 0)) * D;
            if constexpr (FP8) {
                // E4M3 terms: q = (q1 + q2) 2^e, e chosen per head so that
                // the largest |q| 2^-e is in [128, 256).  A bf16 value has 8
                // significant bits; q1 takes the top 4 (rounded) and the
                // remainder, a multiple of the value's last bit no larger
                // than half q1's last bit, fits q2's 4 bits exactly while
                // that last bit is at least E4M3's 2^-9: exact for |q| at
                // least 2^-9 of the head's largest, absolute error below
                // 2^-16 of it otherwise.
                // Lane holds dims 32k + 16j + 4tq .. +3 (k32 B fragment).
                float x[D / 32][2][4];
                float amax = 0.f;
#pragma unroll
                for (int k = 0; k < D / 32; ++k)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint2 r = valid ? __ldg(reinterpret_cast<const uint2 *>(qh + 32 * k + 16 * j + 4 * tq))
                                              : make_uint2(0u, 0u);
                        x[k][j][0] = __uint_as_float(r.x << 16);
                        x[k][j][1] = __uint_as_float(r.x & 0xffff0000u);
                        x[k][j][2] = __uint_as_float(r.y << 16);
                        x[k][j][3] = __uint_as_float(r.y & 0xffff0000u);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            amax = fmaxf(amax, fabsf(x[k][j][e]));
                    }
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                const int ex = amax > 0.f ? max(static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 134, -100)
                                          : 0;
                const float down = __uint_as_float(static_cast<uint32_t>(127 - ex) << 23);
                const float up = __uint_as_float(static_cast<uint32_t>(127 + ex) << 23);
#pragma unroll
                for (int k = 0; k < D / 32; ++k)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        float y[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            y[e] = x[k][j][e] * down;
                        const uint32_t c1 = f32x4_e4m3x4(y[0], y[1], y[2], y[3]);
                        const uint32_t b01 = e4m3x2_lo_f16x2(c1), b23 = e4m3x2_hi_f16x2(c1);
                        qf[2 * k][j] = c1;
                        qf[2 * k + 1][j] = f32x4_e4m3x4(y[0] - f16_lo(b01), y[1] - f16_hi(b01),
                                                        y[2] - f16_lo(b23), y[3] - f16_hi(b23));
                    }
                sl0 = scale_log2 * __shfl_sync(0xffffffffu, up, 4 * h0);
                sl1 = scale_log2 * __shfl_sync(0xffffffffu, up, 4 * h1);
            } else {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    qf[ks][0] = qc[ks][0];
                    qf[ks][1] = qc[ks][1];
                }
            }
        }
        float o[D / 16][4];
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
            o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY;
        // each lane keeps the weight sum of one head (gq & 4 ? h1 : h0; see
        // the reduction below); lanes gq = 0 and 4 write the per-block
        // log2-sum-exps of heads h0 and h1
        const bool wh = gq & 4;
        float lpart = 0.f;
        float *lse_w = nullptr;
        if ((gq & 3) == 0 && (wh ? h1 : h0) < G)
            lse_w = a.w.lse_blk + (static_cast<size_t>(it.l) * g.Hq + kvh * G + (wh ? h1 : h0)) * nb_total + it.lse0;

        for (uint32_t i = 0; i < it.nblk; ++i) {
            mbar_wait(smem_u32(&bars[warp][rg.st_cons]), rg.ph_cons, a.w.err);
            const uint32_t base = ring_u32 + rg.st_cons * T::kStageBytes;

            // S^T = K . Q^T  (rows: 16 tokens, cols: 8 heads)
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            // V fragments (A operand of O^T = V^T P^T), read before the stage is
            // refilled; FP8 keeps the raw codes and converts them at the MMA
            uint32_t va[D / 16][4];
            if constexpr (FP8) {
                // K: an x4 load of 8x8 16-bit tiles over the code bytes gives lane
                // (gq, tq) codes of dims 32k + 4tq..+3 of tokens gq, gq+8 and of
                // dims 32k + 16 + 4tq..+3: the k32 E4M3 A fragment as stored.
                // One accumulator per Q term keeps the MMA chains short.
                float s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int k = 0; k < D / 32; ++k) {
                    const uint32_t row = i8 + 8 * (jm & 1);
                    const uint32_t chunk16 = 2 * k + (jm >> 1);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(base + row * 128 + ((chunk16 ^ (row & 7)) << 4), r0, r1, r2, r3);
                    mma_e4m3(s, r0, r1, r2, r3, qf[2 * k][0], qf[2 * k][1]);
                    mma_e4m3(s2, r0, r1, r2, r3, qf[2 * k + 1][0], qf[2 * k + 1][1]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    s[e] += s2[e];
                // V: a transposing x4 load of 16-bit units gives lane (gq, tq),
                // per tile, tokens 2tq, 2tq+1 x dims 2gq, 2gq+1 of a 16-dim span;
                // tiles: tokens 0-7 / 8-15 x spans 32p / 32p+16
#pragma unroll
                for (int p = 0; p < D / 32; ++p) {
                    const uint32_t row = 16 + i8 + 8 * (jm & 1);
                    const uint32_t chunk16 = 2 * p + (jm >> 1);
                    ldsm_x4_t(base + row * 128 + ((chunk16 ^ (row & 7)) << 4), va[2 * p][0], va[2 * p][1],
                              va[2 * p][2], va[2 * p][3]);
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t h = ks >> 2, c0 = (ks & 3) * 2;
                    const uint32_t row = i8 + 8 * (jm & 1);          // token, K half
                    const uint32_t chunk16 = c0 + (jm >> 1);
                    const uint32_t addr = base + h * T::kBoxBytes + row * 128 + ((chunk16 ^ (row & 7)) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(addr, a0, a1, a2, a3);
                    mma_bf16(s, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
                }
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    const uint32_t h = mt >> 2, c0 = (mt & 3) * 2;
                    const uint32_t row = 16 + i8 + 8 * (jm >> 1);    // V half, token
                    const uint32_t chunk16 = c0 + (jm & 1);
                    const uint32_t addr = base + h * T::kBoxBytes + row * 128 + ((chunk16 ^ (row & 7)) << 4);
                    ldsm_x4_t(addr, va[mt][0], va[mt][1], va[mt][2], va[mt][3]);
                }
            }
            s[0] *= sl0;
            s[1] *= sl1;
            s[2] *= sl0;
            s[3] *= sl1;
            if ((it.b0 + i + 1) * kBlockTokens > it.ntok) {      // the sequence's last block
                const uint32_t tok0 = (it.b0 + i) * kBlockTokens + gq, tok1 = tok0 + 8;
                s[0] = tok0 < it.ntok ? s[0] : -INFINITY;
                s[1] = tok0 < it.ntok ? s[1] : -INFINITY;
                s[2] = tok1 < it.ntok ? s[2] : -INFINITY;
                s[3] = tok1 < it.ntok ? s[3] : -INFINITY;
            }

            // the lanes' maxima are merged only when one of them exceeds the
            // running max; otherwise the running max stands and every rescale
            // factor is 2^0 (the same values as merging, with less work)
            const float lm0 = fmaxf(s[0], s[2]), lm1 = fmaxf(s[1], s[3]);
            const bool moved = __any_sync(0xffffffffu, lm0 > m0 || lm1 > m1);
            // every lane has its K and V fragments: refill the stage
            __syncwarp();
            --rg.inflight;
            if (++rg.st_cons == T::kRing) {
                rg.st_cons = 0;
                rg.ph_cons ^= 1u;
            }
            if (rg.inflight < T::kRing)
                issue_next<D, FP8>(&tmap, g, cur, nxt, have_nxt, c_in_nxt, c_blk, rg, ring_u32, bars[warp], lane);

            float sc0 = 1.f, sc1 = 1.f;
            if (moved) {
                float bm0 = lm0, bm1 = lm1;
#pragma unroll
                for (int x = 4; x < 32; x <<= 1) {
                    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, x));
                    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, x));
                }
                const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
                sc0 = fast_exp2(m0 - mn0);
                sc1 = fast_exp2(m1 - mn1);
                m0 = mn0;
                m1 = mn1;
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    o[mt][0] *= sc0;
                    o[mt][1] *= sc1;
                    o[mt][2] *= sc0;
                    o[mt][3] *= sc1;
                }
            }
            const float p0 = fast_exp2(s[0] - m0), p1 = fast_exp2(s[1] - m1);
            const float p2 = fast_exp2(s[2] - m0), p3 = fast_exp2(s[3] - m1);
            // the block's weight sums over the 8 lanes of each head's column,
            // reduced transposed: lanes gq < 4 end with head h0's, gq >= 4
            // with head h1's
            {
                const float w0 = p0 + p2, w1 = p1 + p3;
                float v = wh ? w1 : w0;
                v += __shfl_xor_sync(0xffffffffu, wh ? w0 : w1, 16);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                lpart = lpart * (wh ? sc1 : sc0) + v;
                if (lse_w)
                    lse_w[i] = (wh ? m1 : m0) + fast_log2(v);
            }
            // P^T as the B operand: transpose the two 8x8 16-bit tiles in registers
            const uint32_t pb0 = movmatrix_t(FP8 ? pack_f16(p0, p1) : pack_bf16(p0, p1));
            const uint32_t pb1 = movmatrix_t(FP8 ? pack_f16(p2, p3) : pack_bf16(p2, p3));
            // O^T += V^T . P^T  (rows: d, cols: 8 heads)
            if constexpr (FP8) {
#pragma unroll
                for (int p = 0; p < D / 32; ++p) {
                    // byte regroup: low half = dim 2gq (tokens 2tq, 2tq+1), high
                    // half = dim 2gq+1; tiles 0/2 feed rows gq/gq+8, 1/3 tokens 8-15
                    const uint32_t t0 = __byte_perm(va[2 * p][0], 0u, 0x3120);
                    const uint32_t t1 = __byte_perm(va[2 * p][1], 0u, 0x3120);
                    const uint32_t t2 = __byte_perm(va[2 * p][2], 0u, 0x3120);
                    const uint32_t t3 = __byte_perm(va[2 * p][3], 0u, 0x3120);
                    mma_f16(o[2 * p], e4m3x2_lo_f16x2(t0), e4m3x2_lo_f16x2(t2), e4m3x2_lo_f16x2(t1),
                            e4m3x2_lo_f16x2(t3), pb0, pb1);
                    mma_f16(o[2 * p + 1], e4m3x2_hi_f16x2(t0), e4m3x2_hi_f16x2(t2), e4m3x2_hi_f16x2(t1),
                            e4m3x2_hi_f16x2(t3), pb0, pb1);
                }
            } else {
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt)
                    mma_bf16(o[mt], va[mt][0], va[mt][1], va[mt][2], va[mt][3], pb0, pb1);
            }

            if (i == claim_at && !have_nxt) {
                // while the ring streams the current item's last blocks
                nxt = prepare_item(a, claim(), lane);
                if constexpr (!FP8)
                    load_q(nxt.it, qn);
                have_nxt = true;
                while (rg.inflight < T::kRing && issue_next<D, FP8>(&tmap, g, cur, nxt, have_nxt, c_in_nxt, c_blk, rg, ring_u32, bars[warp], lane)) {
                }
            }
        }

        // ---- chunk partials ----------------------------------------------
        const float l0 = lpart, l1 = __shfl_xor_sync(0xffffffffu, lpart, 16);   // in lane gq = 0
        const uint32_t part = it.part;
        if (gq == 0) {
            a.w.part_ml[part * kMaxGroup + h0] = make_float2(m0, l0);
            a.w.part_ml[part * kMaxGroup + h1] = make_float2(m1, l1);
        }
        float *po = a.w.part_o + static_cast<size_t>(part) * kMaxGroup * D;
        const float vs = FP8 ? g.v_scale : 1.f;     // values = codes * v_scale
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            const uint32_t d0 = o_dim<FP8>(mt, gq), d1 = o_dim<FP8>(mt, gq + 8);
            po[h0 * D + d0] = o[mt][0] * vs;
            po[h1 * D + d0] = o[mt][1] * vs;
            po[h0 * D + d1] = o[mt][2] * vs;
            po[h1 * D + d1] = o[mt][3] * vs;
        }

        // ---- the next item becomes current ----------------------------------
        if (!have_nxt) {                    // not claimed in the loop: claim now
            nxt = prepare_item(a, claim(), lane);
            if constexpr (!FP8)
                load_q(nxt.it, qn);
        }
        if (c_in_nxt) {
            c_in_nxt = false;               // cursor already inside the new item
        } else {
            c_blk = 0;
        }
        cur = nxt;
        if constexpr (!FP8) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                qc[ks][0] = qn[ks][0];
                qc[ks][1] = qn[ks][1];
            }
        }
        have_nxt = false;
        nxt.it.valid = 0;
        nxt.it.nblk = 0;
        while (cur.it.valid && rg.inflight < T::kRing && issue_next<D, FP8>(&tmap, g, cur, nxt, have_nxt, c_in_nxt, c_blk, rg, ring_u32, bars[warp], lane)) {
        }
    }
}

}  // namespace

size_t decode_smem_bytes(const Geo &g, uint32_t wg)
{
    const size_t per_warp = g.fp8 ? Tile<128, true>::kWarpBytes
                                  : (g.d == 128 ? Tile<128, false>::kWarpBytes : Tile<64, false>::kWarpBytes);
    return wg * per_warp + 1024;   // + alignment slack
}

template <int D, bool FP8>
static int occupancy(const Geo &g, uint32_t wg)
{
    // The attribute is per kernel, shared by every context in the process:
    // always allow the largest configuration (4 warps) so that no context
    // lowers it below what another one launches with.
    int n = 0;
    cudaFuncSetAttribute(decode_kernel<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(decode_smem_bytes(g, 4)));
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<D, FP8>, 32 * wg,
                                                  decode_smem_bytes(g, wg));
    return n;
}

int decode_blocks_per_sm(const Geo &g, uint32_t wg)
{
    if (g.fp8)
        return occupancy<128, true>(g, wg);
    return g.d == 128 ? occupancy<128, false>(g, wg) : occupancy<64, false>(g, wg);
}

cudaError_t launch_decode(const Geo &g, const CUtensorMap &tmap, const Work &w, const uint16_t *q,
                          const int32_t *table, uint32_t n_items, uint32_t wg, int grid,
                          cudaStream_t s)
{
    DecodeArgs a{g, w, q, table, n_items, wg};
    const size_t smem = decode_smem_bytes(g, wg);
    if (g.fp8)
        return launch_pdl(decode_kernel<128, true>, dim3(grid), dim3(32 * wg), smem, s, tmap, a);
    if (g.d == 128)
        return launch_pdl(decode_kernel<128, false>, dim3(grid), dim3(32 * wg), smem, s, tmap, a);
    return launch_pdl(decode_kernel<64, false>, dim3(grid), dim3(32 * wg), smem, s, tmap, a);
}

}  // namespace kvs
