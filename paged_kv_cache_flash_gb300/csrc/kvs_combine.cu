// Split-K combine and block mass (sm_103a).
//
// Sources: "GQA per-head attention as scoring streams" (every (layer, KV head)
// stream contributes to one mass per (sequence, 16-token block)); "KV-Cache
// Offloading for LLM Inference -- Visual Reference" s.4 (the decode output
// over every cached token).
//
//   combine_kernel -- per (sequence, layer, KV head): each CTA recomputes the
//                     heads' log2-sum-exp LSE_h from the chunk partials; CTA
//                     y = 0 merges the output, and the CTAs of the block
//                     ranges turn the per-block log2-sum-exps of their range
//                     into the stream's block masses
//                     sum_h 2^(lse_blk(h, b) - LSE_h).  The merge has a
//                     CTA of its own, or with many short streams shares the
//                     first range's CTA (launch_combine decides).
//   mass_kernel    -- M(b) = 1/(L*Hq) * sum over the L*Hkv streams, in a fixed
//                     order (deterministic); when asked, the thread that
//                     writes M(b) also scores block b's record (score_prep
//                     before the kernel's wait, score_finish after it:
//                     the aggregated mass lands in the 64-byte record).
// Both are launched as programmatic dependents (kvs_pdl.cuh).
#include <type_traits>

#include "kvs_internal.h"
#include "kvs_launch.h"
#include "kvs_pdl.cuh"
#include "kvs_ptx.h"
#include "kvs_score.cuh"

namespace kvs {
namespace {

using namespace ptx;

constexpr uint32_t kMassRange = 2048;   // blocks per combine CTA (stream-mass part)

// split: 1 -> CTA y = 0 merges only and CTA y >= 1 takes block range y - 1;
// 0 -> CTA y takes block range y, and CTA 0 also merges.
template <int D>
__global__ void __launch_bounds__(256, 8) combine_kernel(const Geo g, const Work w, float *out, uint32_t split)
{
    __shared__ float lse_sh[kMaxGroup];
    const DSet *ds = w.dset;
    const uint32_t lane = threadIdx.x & 31, h = threadIdx.x >> 5;
    const uint32_t ci = blockIdx.x / (g.L * g.Hkv);
    const uint32_t rest = blockIdx.x % (g.L * g.Hkv);
    const uint32_t l = rest / g.Hkv, kvh = rest % g.Hkv;
    const DSeq sq = ds->seq[ci];        // the decode set: uploaded before the decode kernel
    pdl_wait();
    pdl_trigger();
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        w.counter[0] = 0;          // ready for the next decode launches
        w.counter[1] = 0;
    }
    const bool merge = blockIdx.y == 0;
    const bool has_range = !split || blockIdx.y > 0;
    const uint32_t r0 = (blockIdx.y - split) * kMassRange;     // unused without a range
    if (!merge && r0 >= sq.nb)
        return;                    // uniform over the CTA
    const uint32_t pb = sq.part_off + (l * g.Hkv + kvh) * sq.nchunk;
    const uint32_t nch = sq.nchunk;
    if (h < g.G) {
        // LSE_h in one pass: each lane keeps a running (max, rescaled sum)
        // over its chunks, then the lanes' pairs are merged
        float m = -INFINITY, sum = 0.f, m_first = -INFINITY;
        for (uint32_t c = lane; c < nch; c += 32) {
            const float2 ml = w.part_ml[(pb + c) * kMaxGroup + h];
            if (c == lane)
                m_first = ml.x;
            const float mn = fmaxf(m, ml.x);
            sum = sum * fast_exp2(m - mn) + ml.y * fast_exp2(ml.x - mn);
            m = mn;
        }
        sum = m == -INFINITY ? 0.f : sum;
#pragma unroll
        for (int x = 16; x > 0; x >>= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, m, x);
            const float so = __shfl_xor_sync(0xffffffffu, sum, x);
            const float mn = fmaxf(m, mo);
            sum = mn == -INFINITY ? 0.f : sum * fast_exp2(m - mn) + so * fast_exp2(mo - mn);
            m = mn;
        }
        const float mmax = m, lsum = sum;
        if (merge) {
            // D / 32 consecutive floats per lane: one 16-byte (D = 128) or
            // 8-byte (D = 64) load per chunk; the chunk maxima of the first
            // 32 chunks come from the lanes that read them above
            using Vec = typename std::conditional<D == 128, float4, float2>::type;
            constexpr int E = D / 32;
            float acc[E];
#pragma unroll
            for (int e = 0; e < E; ++e)
                acc[e] = 0.f;
#pragma unroll 8
            for (uint32_t c = 0; c < nch; ++c) {
                const float mc = c < 32 ? __shfl_sync(0xffffffffu, m_first, c)
                                        : w.part_ml[(pb + c) * kMaxGroup + h].x;
                const float f = fast_exp2(mc - mmax);
                const Vec v = *reinterpret_cast<const Vec *>(
                    w.part_o + (static_cast<size_t>(pb + c) * kMaxGroup + h) * D + lane * E);
                const float *pv = reinterpret_cast<const float *>(&v);
#pragma unroll
                for (int e = 0; e < E; ++e)
                    acc[e] += pv[e] * f;
            }
            const float inv = 1.f / lsum;
            const uint32_t hq = kvh * g.G + h;
            Vec o;
            float *po = reinterpret_cast<float *>(&o);
#pragma unroll
            for (int e = 0; e < E; ++e)
                po[e] = acc[e] * inv;
            *reinterpret_cast<Vec *>(out + ((static_cast<size_t>(ci) * g.L + l) * g.Hq + hq) * D + lane * E) = o;
        }
        if (lane == 0)
            lse_sh[h] = mmax + fast_log2(lsum);
    }
    if (!has_range || r0 >= sq.nb)
        return;                    // uniform over the CTA
    __syncthreads();
    const uint32_t nbt = ds->nb_total;
    const float *lb = w.lse_blk + (static_cast<size_t>(l) * g.Hq + kvh * g.G) * nbt + sq.blk_off;
    float *sm = w.stream_mass + (static_cast<size_t>(l) * g.Hkv + kvh) * nbt + sq.blk_off;
    const uint32_t r1 = min(sq.nb, r0 + kMassRange);
#pragma unroll 4
    for (uint32_t b = r0 + threadIdx.x; b < r1; b += blockDim.x) {
        float acc = 0.f;
#pragma unroll
        for (uint32_t j = 0; j < kMaxGroup; ++j)
            if (j < g.G)
                acc += fast_exp2(lb[static_cast<size_t>(j) * nbt + b] - lse_sh[j]);
        sm[b] = acc;
    }
}

// M(b) = 1/(L*Hq) * sum over the L*Hkv streams of stream_mass(b).  A CTA of
// 1024 threads takes 16 consecutive blocks; thread (i, j) adds the streams
// j, j + 64, ... of block i, and the 64 partial sums of a block are added by
// a fixed tree (deterministic).
constexpr uint32_t kMassBlocks = 16, kMassGroups = 64;

__global__ void __launch_bounds__(1024) mass_kernel(const Geo g, const Work w, float *mass,
                                                    uint32_t nb_total, kvs_record *recs, const ScoreArgs sa,
                                                    uint32_t score)
{
    __shared__ float part[kMassGroups][kMassBlocks + 1];
    const DSet *ds = w.dset;
    const uint32_t i = threadIdx.x % kMassBlocks, j = threadIdx.x / kMassBlocks;
    const uint32_t r = blockIdx.x * kMassBlocks + i;
    uint32_t slot = 0, b = 0, nb = 0;
    uint64_t seq_id = 0, t = 0;
    kvs_record rec;
    ScorePrep prep;
    if (r < nb_total && j == 0) {       // the decode set: uploaded before the decode kernel
        const uint32_t ci = find_seq(&ds->seq[0].blk_off, sizeof(DSeq) / 4, ds->nseq, r);
        slot = ds->seq[ci].slot;
        b = r - ds->seq[ci].blk_off;
        nb = ds->seq[ci].nb;
        seq_id = ds->seq[ci].seq_id;
        t = ds->t;
        // the record: written two or more launches ahead (token append,
        // scoring of earlier steps); the decode and combine kernels write
        // none.  Its mass-free scoring terms (fp64: the decay, the recency
        // division) are taken here, while the combine still runs
        if (score) {
            rec = recs[static_cast<size_t>(slot) * g.mb + b];
            prep = score_prep(sa, rec, seq_id, b, nb, t);
        }
    }
    pdl_wait();
    pdl_trigger();
    const uint32_t LS = g.L * g.Hkv;
    float acc = 0.f;
    if (r < nb_total) {
        // the thread's first 16 streams in one round of loads, added in
        // stream order (as the plain loop would), then any further ones
        float v[16];
#pragma unroll
        for (uint32_t k = 0; k < 16; ++k) {
            const uint32_t s = j + k * kMassGroups;
            v[k] = s < LS ? w.stream_mass[static_cast<size_t>(s) * nb_total + r] : 0.f;
        }
#pragma unroll
        for (uint32_t k = 0; k < 16; ++k)
            acc += v[k];
        for (uint32_t s = j + 16 * kMassGroups; s < LS; s += kMassGroups)
            acc += w.stream_mass[static_cast<size_t>(s) * nb_total + r];
    }
    part[j][i] = acc;
    __syncthreads();
#pragma unroll
    for (uint32_t half = kMassGroups / 2; half > 0; half >>= 1) {
        if (j < half)
            part[j][i] += part[j + half][i];
        __syncthreads();
    }
    if (j == 0 && r < nb_total) {
        const size_t idx = static_cast<size_t>(slot) * g.mb + b;
        const float M = part[0][i] / static_cast<float>(g.L * g.Hq);
        mass[idx] = M;
        if (score)
            score_finish(sa, prep, rec, recs + idx, nb, t, M, w.err);
    }
}

}  // namespace

cudaError_t launch_combine(const Geo &g, const Work &w, float *out, uint32_t nseq, uint32_t max_nb,
                           uint32_t max_nchunk, uint32_t sm_count, cudaStream_t s)
{
    // The merge gets a CTA of its own, beside the block ranges' CTAs, so that
    // the two dependent-load chains run at once, when a stream's merge is long
    // (more than 32 chunks) or when there are no more streams than CTAs fit
    // at once (8 per SM at 32 registers a thread): measured ~3 us less at 8K
    // (640 streams of 12-15 chunks).  With many short streams (the batched
    // workload: 10,240) the extra CTAs only add waves (~10 us more), so the
    // first range's CTA merges too.
    const uint32_t nstreams = nseq * g.L * g.Hkv;
    const uint32_t split = (max_nchunk > 32 || nstreams <= 8 * sm_count) ? 1u : 0u;
    const dim3 grid(nseq * g.L * g.Hkv, split + (max_nb + kMassRange - 1) / kMassRange);
    if (g.d == 128)
        return launch_pdl(combine_kernel<128>, grid, dim3(32 * kMaxGroup), 0, s, g, w, out, split);
    return launch_pdl(combine_kernel<64>, grid, dim3(32 * kMaxGroup), 0, s, g, w, out, split);
}

cudaError_t launch_mass(const Geo &g, const Work &w, float *mass, uint32_t nb_total, kvs_record *recs,
                        const ScoreArgs *score, cudaStream_t s)
{
    const ScoreArgs sa = score ? *score : ScoreArgs{};
    return launch_pdl(mass_kernel, dim3((nb_total + kMassBlocks - 1) / kMassBlocks), dim3(1024), 0, s, g, w,
                      mass, nb_total, recs, sa, score ? 1u : 0u);
}

}  // namespace kvs
