// Block-level kernels: append into pages, EMA/priority/tier scoring,
// selection (threshold compaction and lowest-fraction radix select), page
// gather into the staging ring, and table/record patches for demote/readmit.
//
// Sources: "KV-Cache Offloading for LLM Inference -- Visual Reference" s.11
// (EMA rule), s.12 (priority P, tier thresholds 0.3 / 0.6); "GQA per-head
// attention as scoring streams" (64-byte per-block state, identity key kept
// across eviction); "LLM KV cache offload" (block tables, pinned-host
// staging); "RETRACTIONS" s.3 (exact victim selection, audited by brute force).
#include <algorithm>
#include <cstring>

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kvs_internal.h"
#include "kvs_launch.h"
#include "kvs_pdl.cuh"
#include "kvs_score.cuh"

namespace kvs {
namespace {

// ----------------------------------------------------------------- append
// One 16-byte vector of a page row from the token-major bf16 source row:
// 8 bf16 values as they are, or (FP8 pages) 16 values quantised to E4M3 codes,
// code = e4m3(x / scale) with an IEEE fp32 division, nearest code, saturating.
__device__ __forceinline__ uint4 page_vec_from_bf16(const Geo &g, const uint16_t *src_row, uint32_t v16,
                                                    float scale)
{
    if (!g.fp8)
        return __ldg(reinterpret_cast<const uint4 *>(src_row) + v16);
    const uint4 a = __ldg(reinterpret_cast<const uint4 *>(src_row) + 2 * v16);
    const uint4 b = __ldg(reinterpret_cast<const uint4 *>(src_row) + 2 * v16 + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t packed = 0;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const uint32_t word = w[2 * q + r];
            const float x0 = __fdiv_rn(__uint_as_float(word << 16), scale);
            const float x1 = __fdiv_rn(__uint_as_float(word & 0xffff0000u), scale);
            const __nv_fp8x2_storage_t c =
                __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
            packed |= static_cast<uint32_t>(c) << (16 * r);
        }
        out[q] = packed;
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

__device__ __forceinline__ uint8_t *page_row(const Geo &g, uint8_t *pool, int32_t page, uint32_t l,
                                             uint32_t kv, uint32_t h, uint32_t slot)
{
    const uint64_t elem = g.fp8 ? 1 : 2;
    return pool + static_cast<uint64_t>(page) * g.page_bytes +
           (((static_cast<uint64_t>(l) * 2 + kv) * g.Hkv + h) * kBlockTokens + slot) * g.d * elem;
}

// One thread moves 16 bytes.  Rows are (token slot, layer, K/V, KV head) of
// d bf16 values; slots of the last touched block past the appended tokens
// are zero-filled.  Thread-blocks past the row range initialise the records
// of newly opened blocks and their table entries.
__global__ void append_kernel(const Geo g, const AppendArgs a, uint64_t rows_total,
                              uint32_t vec_per_row)
{
    const uint64_t tid = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const uint64_t nvec = rows_total * vec_per_row;
    if (tid < nvec) {
        const uint64_t row = tid / vec_per_row;
        const uint32_t v16 = static_cast<uint32_t>(tid % vec_per_row);
        // row = ((slot_pos * L + l) * 2 + kv) * Hkv + h, slot_pos from p0
        const uint32_t h = row % g.Hkv;
        uint64_t r2 = row / g.Hkv;
        const uint32_t kv = r2 % 2;
        r2 /= 2;
        const uint32_t l = r2 % g.L;
        const uint64_t rel = r2 / g.L;                  // token position - p0
        const uint64_t pos = a.p0 + rel;
        const uint32_t blk = static_cast<uint32_t>(pos / kBlockTokens);
        const uint32_t slot_in = static_cast<uint32_t>(pos % kBlockTokens);
        const int32_t page = a.pages[blk - a.first_blk];
        uint4 val = make_uint4(0, 0, 0, 0);
        if (rel < a.n) {
            const uint16_t *src = (kv == 0 ? a.k : a.v) + ((rel * g.L + l) * g.Hkv + h) * g.d;
            val = page_vec_from_bf16(g, src, v16, kv == 0 ? g.k_scale : g.v_scale);
        }
        uint8_t *dst = page_row(g, reinterpret_cast<uint8_t *>(a.pool), page, l, kv, h, slot_in);
        reinterpret_cast<uint4 *>(dst)[v16] = val;
    } else {
        const uint64_t j = tid - nvec;                  // new-block index
        const uint32_t nnew = a.first_blk + a.nblk - a.first_new;
        if (j < a.nblk)
            a.page_clean[a.pages[j]] = 0;               // page bytes change
        if (j < nnew) {
            const uint32_t b = a.first_new + static_cast<uint32_t>(j);
            const size_t idx = static_cast<size_t>(a.slot) * g.mb + b;
            kvs_record r;
            r.key.seq_id = a.seq_id;
            r.key.block_idx = b;
            r.score = 0.0;
            r.last_touch = a.t_create;
            r.count = 0;
            r.tier = 255;
            r.flags = 0;
            r.pad0 = 0;
            r.prio = 0.0;
            r.mass = 0.f;
            for (int q = 0; q < 4; ++q)
                r.reserved[q] = 0;
            r.lrfu = 0.0;
            a.records[idx] = r;
            a.table[idx] = a.pages[b - a.first_blk];
        }
    }
}

// One token per sequence: thread -> (sequence by binary search on row_off,
// row, 16-byte vector).  Row 0 of a sequence's rows holds the token; rows of
// later slots (a freshly opened block) are zero-filled.  The first threads
// past the row range write the records and table entries of fresh blocks.
// sa: the per-sequence entries in device memory, or null when they come in
// the parameters (inl, at most kStepInline of them).
__global__ void append_step_kernel(const Geo g, const uint16_t *k, const uint16_t *v, uint16_t *pool,
                                   int32_t *table, kvs_record *records, uint8_t *page_clean,
                                   const StepAppend *sa_dev, const __grid_constant__ StepAppendInline inl,
                                   uint32_t nseq, uint32_t rows_total, uint32_t vec_per_row, uint64_t t_create)
{
    pdl_wait();                 // the pages, table and records may still be read by earlier kernels
    pdl_trigger();
    const StepAppend *sa = sa_dev ? sa_dev : inl.e;
    const uint64_t tid = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const uint64_t nvec = static_cast<uint64_t>(rows_total) * vec_per_row;
    if (tid < nvec) {
        const uint32_t row = static_cast<uint32_t>(tid / vec_per_row);
        const uint32_t v16 = static_cast<uint32_t>(tid % vec_per_row);
        uint32_t lo = 0, hi = nseq;
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) >> 1;
            if (sa[mid].row_off <= row)
                lo = mid;
            else
                hi = mid;
        }
        const StepAppend a = sa[lo];
        const uint32_t r = row - a.row_off;
        // r = ((slot_rel * L + l) * 2 + kv) * Hkv + h
        const uint32_t h = r % g.Hkv;
        uint32_t r2 = r / g.Hkv;
        const uint32_t kv = r2 % 2;
        r2 /= 2;
        const uint32_t l = r2 % g.L;
        const uint32_t rel = r2 / g.L;
        const uint32_t slot_in = a.pos % kBlockTokens + rel;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (rel == 0) {
            const uint16_t *src = (kv == 0 ? k : v) + ((static_cast<size_t>(lo) * g.L + l) * g.Hkv + h) * g.d;
            val = page_vec_from_bf16(g, src, v16, kv == 0 ? g.k_scale : g.v_scale);
        }
        uint8_t *dst = page_row(g, reinterpret_cast<uint8_t *>(pool), a.page, l, kv, h, slot_in);
        reinterpret_cast<uint4 *>(dst)[v16] = val;
    } else {
        const uint64_t i = tid - nvec;
        if (i < nseq) {
            const StepAppend a = sa[i];
            page_clean[a.page] = 0;
            if (a.fresh) {
                const uint32_t b = a.pos / kBlockTokens;
                const size_t idx = static_cast<size_t>(a.slot) * g.mb + b;
                kvs_record rec;
                rec.key.seq_id = a.seq_id;
                rec.key.block_idx = b;
                rec.score = 0.0;
                rec.last_touch = t_create;
                rec.count = 0;
                rec.tier = 255;
                rec.flags = 0;
                rec.pad0 = 0;
                rec.prio = 0.0;
                rec.mass = 0.f;
                for (int q = 0; q < 4; ++q)
                    rec.reserved[q] = 0;
                rec.lrfu = 0.0;
                records[idx] = rec;
                table[idx] = a.page;
            }
        }
    }
}

// ----------------------------------------------------------------- scoring
__device__ __forceinline__ uint32_t find_sorted(const DSet *ds, uint32_t r)
{
    uint32_t lo = 0, hi = ds->nseq;
    while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        if (ds->seq[mid].srt_off <= r)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// One thread per record of the decode set (record order: ascending seq_id,
// then block); the scoring itself is score_record (kvs_score.cuh).
__global__ void score_kernel(const Geo g, const Work w, kvs_record *recs, const float *mass,
                             const ScoreArgs sa, uint32_t nb_total)
{
    const uint32_t r = blockIdx.x * blockDim.x + threadIdx.x;
    const DSet *ds = w.dset;
    // the decode set was uploaded before the decode kernel: read it while the
    // mass is being finished
    DSeq sq{};
    uint32_t b = 0;
    uint64_t t = 0;
    if (r < nb_total) {
        const uint32_t si = find_sorted(ds, r);
        sq = ds->seq[ds->seq[si].srt_ci];
        b = r - ds->seq[si].srt_off;
        t = ds->t;
    }
    pdl_wait();
    pdl_trigger();
    if (r >= nb_total)
        return;
    const size_t idx = static_cast<size_t>(sq.slot) * g.mb + b;
    score_record(sa, recs, idx, sq.seq_id, b, sq.nb, t, mass[idx], w.err);
}

// ---------------------------------------------------------------- selection
constexpr int kSelThreads = 256;
constexpr int kSelPerThread = 4;
constexpr int kSelTile = kSelThreads * kSelPerThread;

// Record-array index of record r of the decode set (record order), with its
// sequence slot, block and token count (each optional).  Reads the decode set
// only.
__device__ __forceinline__ size_t rec_index(const Geo &g, const DSet *ds, uint32_t r, uint32_t *slot_out,
                                            uint32_t *b_out, uint32_t *ntok_out)
{
    const uint32_t si = find_sorted(ds, r);
    const DSeq &sq = ds->seq[ds->seq[si].srt_ci];
    const uint32_t b = r - ds->seq[si].srt_off;
    if (slot_out)
        *slot_out = sq.slot;
    if (b_out)
        *b_out = b;
    if (ntok_out)
        *ntok_out = sq.ntok;
    return static_cast<size_t>(sq.slot) * g.mb + b;
}

__device__ __forceinline__ const kvs_record &rec_at(const Geo &g, const DSet *ds,
                                                    const kvs_record *recs, uint32_t r,
                                                    uint32_t *slot_out, uint32_t *b_out,
                                                    uint32_t *ntok_out = nullptr)
{
    const uint32_t si = find_sorted(ds, r);
    const DSeq &sq = ds->seq[ds->seq[si].srt_ci];
    const uint32_t b = r - ds->seq[si].srt_off;
    *slot_out = sq.slot;
    *b_out = b;
    if (ntok_out)
        *ntok_out = sq.ntok;
    return recs[static_cast<size_t>(sq.slot) * g.mb + b];
}

// Natural logarithm of a positive normal double from its series definition
// (Abramowitz and Stegun, Handbook of Mathematical Functions, 4.1.27):
// x = m 2^e with m in [sqrt(1/2), sqrt(2)); s = (m - 1)/(m + 1), z = s*s;
// ln m = 2 artanh(s) = 2 s (1 + z/3 + z^2/5 + ... + z^11/23), the bracket by
// Horner's rule from the 1/23 term down; ln x = e ln2 + ln m.  |s| < 0.172,
// so the cut-off term is below 1e-20 of the first.  Each step is one
// correctly rounded fp64 operation in a fixed order (explicit round-to-nearest
// intrinsics, no fused multiply-add), so the same steps give the same bits on
// any IEEE machine: near-equal LRFU keys then order the same way everywhere.
__device__ __forceinline__ double ln_series(double x)
{
    constexpr double kLn2 = 0x1.62e42fefa39efp-1;        // the double nearest ln 2
    constexpr double kSqrtHalf = 0x1.6a09e667f3bcdp-1;   // the double nearest sqrt(1/2)
    const long long bits = __double_as_longlong(x);
    int e = static_cast<int>((bits >> 52) & 0x7ff) - 1022;              // x = m 2^e, m in [1/2, 1)
    double m = __longlong_as_double((bits & 0x000fffffffffffffLL) | 0x3fe0000000000000LL);
    if (m < kSqrtHalf) {
        m = __dmul_rn(m, 2.0);
        e -= 1;
    }
    const double s = __ddiv_rn(__dsub_rn(m, 1.0), __dadd_rn(m, 1.0));
    const double z = __dmul_rn(s, s);
    double h = 1.0 / 23.0;
    h = __dadd_rn(1.0 / 21.0, __dmul_rn(z, h));
    h = __dadd_rn(1.0 / 19.0, __dmul_rn(z, h));
    h = __dadd_rn(1.0 / 17.0, __dmul_rn(z, h));
    h = __dadd_rn(1.0 / 15.0, __dmul_rn(z, h));
    h = __dadd_rn(1.0 / 13.0, __dmul_rn(z, h));
    h = __dadd_rn(1.0 / 11.0, __dmul_rn(z, h));
    h = __dadd_rn(1.0 / 9.0, __dmul_rn(z, h));
    h = __dadd_rn(1.0 / 7.0, __dmul_rn(z, h));
    h = __dadd_rn(1.0 / 5.0, __dmul_rn(z, h));
    h = __dadd_rn(1.0 / 3.0, __dmul_rn(z, h));
    h = __dadd_rn(1.0, __dmul_rn(z, h));
    return __dadd_rn(__dmul_rn(static_cast<double>(e), kLn2), __dmul_rn(2.0, __dmul_rn(s, h)));
}

// Slope of the LRFU key per step of the touch time: -ln(1 - alpha).
__device__ __forceinline__ double lrfu_slope(double alpha)
{
    return -ln_series(__dsub_rn(1.0, alpha));
}

// 64-bit order key of a record for LOWFRAC (P >= 0: its bits order like P)
// and LRFU (K = ln lrfu + last_touch * c with c = lrfu_slope(alpha), -inf
// for a block never touched, mapped to bits that order like K: negative
// values complemented, others with the top bit set).
__device__ __forceinline__ uint64_t sel_key(int mode, const kvs_record &rec, double c)
{
    if (mode != KVS_SELECT_LRFU)
        return static_cast<uint64_t>(__double_as_longlong(rec.prio));
    const double K = rec.lrfu > 0.0
                         ? __dadd_rn(ln_series(rec.lrfu), __dmul_rn(static_cast<double>(rec.last_touch), c))
                         : -__longlong_as_double(0x7ff0000000000000LL);
    const uint64_t u = static_cast<uint64_t>(__double_as_longlong(K));
    return (u >> 63) ? ~u : (u | (uint64_t(1) << 63));
}

__device__ __forceinline__ bool picked(int mode, const kvs_record &rec, uint32_t r,
                                       const uint64_t *thr, double c)
{
    if (mode == KVS_SELECT_THRESH)
        return rec.tier == 2;
    // composite key (order key, record index)
    const uint64_t pb = sel_key(mode, rec, c);
    return pb < thr[0] || (pb == thr[0] && r <= thr[1]);
}

// Counts picked records per tile of kSelTile records.
__global__ void __launch_bounds__(kSelThreads)
    select_count_kernel(const Geo g, const Work w, const kvs_record *recs, int mode, double alpha,
                        uint32_t nb_total)
{
    const double lrfu_c = mode == KVS_SELECT_LRFU ? lrfu_slope(alpha) : 0.0;
    __shared__ uint32_t wsum[kSelThreads / 32];
    const DSet *ds = w.dset;
    size_t idx[kSelPerThread];
    for (int q = 0; q < kSelPerThread; ++q) {
        const uint32_t r = blockIdx.x * kSelTile + threadIdx.x * kSelPerThread + q;
        idx[q] = r < nb_total ? rec_index(g, ds, r, nullptr, nullptr, nullptr) : 0;
    }
    pdl_wait();                 // records and the threshold come from earlier kernels
    pdl_trigger();
    uint32_t c = 0;
    for (int q = 0; q < kSelPerThread; ++q) {
        const uint32_t r = blockIdx.x * kSelTile + threadIdx.x * kSelPerThread + q;
        if (r < nb_total)
            c += picked(mode, recs[idx[q]], r, w.sel_thr, lrfu_c) ? 1u : 0u;
    }
    for (int x = 16; x > 0; x >>= 1)
        c += __shfl_xor_sync(0xffffffffu, c, x);
    if ((threadIdx.x & 31) == 0)
        wsum[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
        for (int q = 0; q < kSelThreads / 32; ++q)
            t += wsum[q];
        w.tile_cnt[blockIdx.x] = t;
    }
}

// Writes picked records in record order: key, page and record index.
// out: optional direct outputs -- the caller's key list (ids, first ids_cap
// entries) and, through its device mapping, a host word for the count.
__global__ void __launch_bounds__(kSelThreads)
    select_scatter_kernel(const Geo g, const Work w, const kvs_record *recs, const int32_t *table,
                          int mode, double alpha, uint32_t nb_total, uint32_t ntiles, uint32_t count_pages,
                          const SelectOut out)
{
    const double lrfu_c = mode == KVS_SELECT_LRFU ? lrfu_slope(alpha) : 0.0;
    __shared__ uint32_t wpre[kSelThreads / 32];
    __shared__ uint32_t base_sh;
    const DSet *ds = w.dset;
    uint32_t bs[kSelPerThread], nts[kSelPerThread];
    size_t idx[kSelPerThread];
    for (int q = 0; q < kSelPerThread; ++q) {
        const uint32_t r = blockIdx.x * kSelTile + threadIdx.x * kSelPerThread + q;
        idx[q] = r < nb_total ? rec_index(g, ds, r, nullptr, &bs[q], &nts[q]) : 0;
    }
    pdl_wait();                 // tile counts and records come from earlier kernels
    pdl_trigger();
    if (threadIdx.x == 0) {
        // one tile: no count kernel ran; the count is this CTA's own total
        uint32_t base = 0;
        for (uint32_t q = 0; q < blockIdx.x; ++q)
            base += w.tile_cnt[q];
        base_sh = base;
        if (ntiles > 1 && blockIdx.x == ntiles - 1) {
            *w.sel_count = base + w.tile_cnt[blockIdx.x];
            if (out.count_host)
                *out.count_host = base + w.tile_cnt[blockIdx.x];
        }
    }
    // records and their table entries (same [slot][block] index) in one round
    bool pk[kSelPerThread];
    kvs_record rv[kSelPerThread];
    int32_t pages[kSelPerThread];
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q) {
        const uint32_t r = blockIdx.x * kSelTile + threadIdx.x * kSelPerThread + q;
        if (r < nb_total) {
            rv[q] = recs[idx[q]];
            pages[q] = table[idx[q]];
        }
    }
    uint32_t c = 0;
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q) {
        const uint32_t r = blockIdx.x * kSelTile + threadIdx.x * kSelPerThread + q;
        pk[q] = r < nb_total && picked(mode, rv[q], r, w.sel_thr, lrfu_c);
        c += pk[q] ? 1u : 0u;
    }
    // exclusive scan of c over the block
    const uint32_t lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t inc = c;
    for (int x = 1; x < 32; x <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc, x);
        if (lane >= static_cast<uint32_t>(x))
            inc += y;
    }
    if (lane == 31)
        wpre[wid] = inc;
    __syncthreads();
    uint32_t wbase = 0;
    for (uint32_t q = 0; q < wid; ++q)
        wbase += wpre[q];
    if (ntiles == 1 && threadIdx.x == 0) {
        uint32_t total = 0;
        for (uint32_t q = 0; q < kSelThreads / 32; ++q)
            total += wpre[q];
        *w.sel_count = total;
        if (out.count_host)
            *out.count_host = total;
    }
    uint32_t pos = base_sh + wbase + inc - c;
#pragma unroll
    for (int q = 0; q < kSelPerThread; ++q) {
        if (!pk[q])
            continue;
        const uint32_t r = blockIdx.x * kSelTile + threadIdx.x * kSelPerThread + q;
        const int32_t page = pages[q];
        w.sel_ids[pos] = rv[q].key;
        if (out.ids && pos < out.ids_cap)
            out.ids[pos] = rv[q].key;
        w.sel_recs[pos] = rv[q];
        w.sel_pages[pos] = page;
        w.sel_recidx[pos] = r;
        w.sel_full[pos] = (bs[q] + 1) * kBlockTokens <= nts[q] ? 1 : 0;
        if (count_pages && page >= 0) {
            // for the gather plan: listed references and first list position per page
            atomicAdd(&w.page_cnt[page], 1u);
            atomicMin(&w.page_first[page], pos);
        }
        ++pos;
    }
}

// k-th smallest composite key (order key of the mode, record index), k >= 1,
// by an 8-bit radix descent over the 96-bit key.  One block of 1024 threads.
__global__ void __launch_bounds__(1024)
    radix_select_kernel(const Geo g, const Work w, const kvs_record *recs, uint32_t nb_total,
                        uint32_t k, int mode, double alpha)
{
    const double c = mode == KVS_SELECT_LRFU ? lrfu_slope(alpha) : 0.0;
    __shared__ uint32_t hist[256];
    __shared__ uint64_t pre_p;
    __shared__ uint32_t pre_r;
    __shared__ uint32_t remaining;
    const DSet *ds = w.dset;
    pdl_wait();                 // records come from the scoring kernel
    pdl_trigger();
    if (threadIdx.x == 0) {
        pre_p = 0;
        pre_r = 0;
        remaining = k;
    }
    // 8 passes over the prio bits, then 4 over the record index
    for (int pass = 0; pass < 12; ++pass) {
        for (uint32_t q = threadIdx.x; q < 256; q += blockDim.x)
            hist[q] = 0;
        __syncthreads();
        const uint64_t pp = pre_p;
        const uint32_t pr = pre_r;
        for (uint32_t r = threadIdx.x; r < nb_total; r += blockDim.x) {
            uint32_t slot, b;
            const kvs_record &rec = rec_at(g, ds, recs, r, &slot, &b);
            const uint64_t pbits = sel_key(mode, rec, c);
            uint32_t digit;
            bool match;
            if (pass < 8) {
                const int sh = 56 - 8 * pass;
                const uint64_t mask = pass == 0 ? 0ull : (~0ull << (sh + 8));
                match = (pbits & mask) == pp;
                digit = static_cast<uint32_t>(pbits >> sh) & 0xffu;
            } else {
                const int sh = 24 - 8 * (pass - 8);
                const uint32_t mask = pass == 8 ? 0u : (~0u << (sh + 8));
                match = pbits == pp && (r & mask) == pr;
                digit = (r >> sh) & 0xffu;
            }
            if (match)
                atomicAdd(&hist[digit], 1u);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t rem = remaining, dsel = 255;
            for (uint32_t q = 0; q < 256; ++q) {
                if (hist[q] >= rem) {
                    dsel = q;
                    break;
                }
                rem -= hist[q];
            }
            remaining = rem;
            if (pass < 8)
                pre_p |= static_cast<uint64_t>(dsel) << (56 - 8 * pass);
            else
                pre_r |= dsel << (24 - 8 * (pass - 8));
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        w.sel_thr[0] = pre_p;
        w.sel_thr[1] = pre_r;
    }
}

// --------------------------------------------------------------- gather plan
// Exclusive scan of one flag per thread over a 1024-thread block; returns the
// thread's position and writes the block total to *total.
__device__ __forceinline__ uint32_t block_scan_1024(uint32_t f, uint32_t *wsum, uint32_t *total)
{
    const uint32_t lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t inc = f;
    for (int x = 1; x < 32; x <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc, x);
        if (lane >= static_cast<uint32_t>(x))
            inc += y;
    }
    if (lane == 31)
        wsum[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        uint32_t v = wsum[lane], vi = v;
        for (int x = 1; x < 32; x <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, vi, x);
            if (lane >= static_cast<uint32_t>(x))
                vi += y;
        }
        wsum[lane] = vi - v;            // exclusive warp offsets
        if (lane == 31)
            wsum[32] = vi;
    }
    __syncthreads();
    const uint32_t pos = wsum[wid] + inc - f;
    *total = wsum[32];
    __syncthreads();
    return pos;
}

// Selection and gather plan of a set of at most one tile (kSelOneTile
// records) in one CTA: thread r takes record r (record order), the picks are
// placed by a block scan (list order = record order among the picks), and
// each picking thread then plans its own list entry -- a page is gathered at
// its first entry once every record that references it is listed -- as
// plan_kernel does.  A page referenced once (the common case: no shared
// prefix) needs no counting: its one entry leads.  Pages of several
// references are counted with atomics before the first scan, whose barriers
// order them before the counts are read; the first entry is the one of the
// smallest record index, which is the smallest list position.  Outputs as
// select_scatter_kernel + plan_kernel: the list, its records and pages, the
// plan, the slots, the counts (readback and, through its device mapping,
// out.count_host), the per-page counters back at 0 / ~0.
constexpr uint32_t kSelOneTile = 1024;

__global__ void __launch_bounds__(kSelOneTile)
    select_plan_kernel(const Geo g, const Work w, const kvs_record *recs, const int32_t *table, int mode,
                       double alpha, uint32_t nb_total, uint32_t mirror, const SelectOut out)
{
    __shared__ uint32_t wsum[33];
    const double lrfu_c = mode == KVS_SELECT_LRFU ? lrfu_slope(alpha) : 0.0;
    const DSet *ds = w.dset;
    const uint32_t r = threadIdx.x;
    uint32_t b = 0, nt = 0;
    size_t idx = 0;
    if (r < nb_total)
        idx = rec_index(g, ds, r, nullptr, &b, &nt);
    pdl_wait();                 // records (and the LOWFRAC threshold) come from earlier kernels
    pdl_trigger();
    kvs_record rec;
    int32_t page = -1;
    uint32_t ref = 0, clean = 1;
    bool pk = false;
    if (r < nb_total) {
        rec = recs[idx];
        page = table[idx];
        if (page >= 0) {
            ref = w.dev_refcnt[page];
            clean = w.page_clean[page];
        }
        pk = picked(mode, rec, r, w.sel_thr, lrfu_c);
    }
    const bool shared = pk && page >= 0 && ref != 1;
    if (shared) {
        atomicAdd(&w.page_cnt[page], 1u);
        atomicMin(&w.page_first[page], r);
    }
    uint32_t nsel;
    const uint32_t pos = block_scan_1024(pk ? 1u : 0u, wsum, &nsel);   // its barriers order the atomics
    if (pk) {
        w.sel_ids[pos] = rec.key;
        if (out.ids && pos < out.ids_cap)
            out.ids[pos] = rec.key;
        w.sel_recs[pos] = rec;
        w.sel_pages[pos] = page;
        w.sel_recidx[pos] = r;
        w.sel_full[pos] = (b + 1) * kBlockTokens <= nt ? 1 : 0;
    }
    if (threadIdx.x == 0)
        *w.sel_count = nsel;
    // ---- plan: each picking thread decides for its own list entry ----
    bool whole = pk && page >= 0;            // every reference of the page is listed
    uint32_t lead = whole ? 1u : 0u;
    if (shared) {
        const uint32_t cnt = __ldcg(&w.page_cnt[page]);
        whole = cnt == ref;
        lead = (whole && __ldcg(&w.page_first[page]) == r) ? 1u : 0u;
    }
    const uint32_t dirty = (lead && mirror && !clean) ? 1u : 0u;
    uint32_t tot;
    const uint32_t ex = block_scan_1024(lead | (dirty << 16), wsum, &tot);
    if (lead) {
        const uint32_t ppos = ex & 0xffffu;
        w.plan_pages[ppos] = page;
        if (!mirror)
            w.page_pos[page] = static_cast<int32_t>(ppos);
    }
    if (dirty) {
        w.readback[4 + (ex >> 16)] = static_cast<uint32_t>(page);
        w.page_clean[page] = (b + 1) * kBlockTokens <= nt ? 1 : 0;
    }
    if (!mirror)
        __syncthreads();        // page_pos of every leader is written
    if (pk) {
        const int32_t v = whole ? (mirror ? page : __ldcg(&w.page_pos[page])) : -1;
        w.plan_slot[pos] = v;
        if (out.slots && pos < out.ids_cap)
            out.slots[pos] = v;
    }
    if (shared) {               // every read of the counters was before the second scan's barriers
        w.page_cnt[page] = 0;
        w.page_first[page] = 0xffffffffu;
    }
    if (threadIdx.x == 0) {
        w.readback[0] = nsel;
        w.readback[1] = tot & 0xffffu;
        w.readback[2] = tot >> 16;
        w.readback[3] = 0;
        if (out.count_host) {
            out.count_host[0] = nsel;
            out.count_host[1] = tot & 0xffffu;
            out.count_host[2] = tot >> 16;
            out.count_host[3] = 0;
        }
    }
}

// ------------------------------------------------------------- prefetch plan
// Order key of a demoted block: class in the top two bits (0 anchor zone,
// 1 recent window, 2 other), then the blend descending as 1.0's bits minus
// the blend's bits (blend in [0, 1], so the difference fits 62 bits and
// orders exactly like the blend, reversed).
constexpr uint64_t kOneBits = 0x3FF0000000000000ull;
constexpr int64_t kAnchorLastPos = 100;     // anchor zone: positions 0..100
constexpr int64_t kRecentWindow = 200;      // recent window: m-200..m-1

__device__ __forceinline__ uint64_t prefetch_key(const PrefCand &c)
{
    const int64_t first = static_cast<int64_t>(c.block) * kBlockTokens;
    const int64_t last = first + kBlockTokens - 1;
    const int64_t m = c.ntok;
    const uint64_t cls = first <= kAnchorLastPos ? 0u : (last >= m - kRecentWindow ? 1u : 2u);
    const int64_t dist = max(static_cast<int64_t>(0), (m - 1) - last);
    const double rope = __ddiv_rn(1.0, __dadd_rn(1.0, __ddiv_rn(static_cast<double>(dist), 100.0)));
    const double blend = __dadd_rn(__dmul_rn(0.6, rope), __dmul_rn(0.4, c.ema));
    uint64_t bits = static_cast<uint64_t>(__double_as_longlong(blend));
    bits = bits > kOneBits ? kOneBits : bits;
    return (cls << 62) | (kOneBits - bits);
}

// One block of 1024 threads: keys of the n candidates, the k-th smallest
// (key, index) by an 8-bit radix descent (when k < n), the k smallest
// compacted in index order, then a bitonic sort of them in shared memory.
__global__ void __launch_bounds__(1024)
    prefetch_plan_kernel(const PrefCand *cand, uint32_t n, uint32_t k, uint64_t *keys,
                         uint64_t *out_key, uint32_t *out_idx)
{
    extern __shared__ __align__(16) uint8_t psm[];
    uint64_t *skey = reinterpret_cast<uint64_t *>(psm);
    uint32_t *sidx = reinterpret_cast<uint32_t *>(psm + KVS_PREFETCH_MAX * sizeof(uint64_t));
    __shared__ uint32_t hist[256];
    __shared__ uint32_t wsum[33];
    __shared__ uint64_t pre_k;
    __shared__ uint32_t pre_i, remaining, base;

    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x)
        keys[i] = prefetch_key(cand[i]);
    if (threadIdx.x == 0) {
        pre_k = 0;
        pre_i = 0;
        remaining = k;
        base = 0;
    }
    __syncthreads();
    uint64_t tk = ~0ull;
    uint32_t ti = ~0u;
    if (k < n) {
        // 8 passes over the key bits, then 4 over the candidate index
        for (int pass = 0; pass < 12; ++pass) {
            for (uint32_t q = threadIdx.x; q < 256; q += blockDim.x)
                hist[q] = 0;
            __syncthreads();
            const uint64_t pk = pre_k;
            const uint32_t pi = pre_i;
            for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) {
                const uint64_t key = keys[i];
                uint32_t digit;
                bool match;
                if (pass < 8) {
                    const int sh = 56 - 8 * pass;
                    const uint64_t mask = pass == 0 ? 0ull : (~0ull << (sh + 8));
                    match = (key & mask) == pk;
                    digit = static_cast<uint32_t>(key >> sh) & 0xffu;
                } else {
                    const int sh = 24 - 8 * (pass - 8);
                    const uint32_t mask = pass == 8 ? 0u : (~0u << (sh + 8));
                    match = key == pk && (i & mask) == pi;
                    digit = (i >> sh) & 0xffu;
                }
                if (match)
                    atomicAdd(&hist[digit], 1u);
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                uint32_t rem = remaining, dsel = 255;
                for (uint32_t q = 0; q < 256; ++q) {
                    if (hist[q] >= rem) {
                        dsel = q;
                        break;
                    }
                    rem -= hist[q];
                }
                remaining = rem;
                if (pass < 8)
                    pre_k |= static_cast<uint64_t>(dsel) << (56 - 8 * pass);
                else
                    pre_i |= dsel << (24 - 8 * (pass - 8));
            }
            __syncthreads();
        }
        tk = pre_k;
        ti = pre_i;
    }
    // the k entries with (key, index) <= (tk, ti), in index order
    for (uint32_t t0 = 0; t0 < n; t0 += blockDim.x) {
        const uint32_t i = t0 + threadIdx.x;
        uint64_t key = 0;
        uint32_t f = 0;
        if (i < n) {
            key = keys[i];
            f = (key < tk || (key == tk && i <= ti)) ? 1u : 0u;
        }
        uint32_t tot;
        const uint32_t pos = base + block_scan_1024(f, wsum, &tot);
        if (f && pos < KVS_PREFETCH_MAX) {
            skey[pos] = key;
            sidx[pos] = i;
        }
        __syncthreads();
        if (threadIdx.x == 0)
            base += tot;
        __syncthreads();
    }
    uint32_t P = 1;
    while (P < k)
        P <<= 1;
    for (uint32_t i = k + threadIdx.x; i < P; i += blockDim.x) {
        skey[i] = ~0ull;
        sidx[i] = ~0u;
    }
    __syncthreads();
    for (uint32_t size = 2; size <= P; size <<= 1)
        for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
            for (uint32_t i = threadIdx.x; i < P; i += blockDim.x) {
                const uint32_t j = i ^ stride;
                if (j > i) {
                    const bool up = (i & size) == 0;
                    const uint64_t ki = skey[i], kj = skey[j];
                    const uint32_t ii = sidx[i], ij = sidx[j];
                    const bool gt = ki > kj || (ki == kj && ii > ij);
                    if (gt == up) {
                        skey[i] = kj;
                        skey[j] = ki;
                        sidx[i] = ij;
                        sidx[j] = ii;
                    }
                }
            }
            __syncthreads();
        }
    for (uint32_t i = threadIdx.x; i < k; i += blockDim.x) {
        out_key[i] = skey[i];
        out_idx[i] = sidx[i];
    }
}

// Gather plan of the selected list, one block of 1024 threads, from the
// per-page counts select_scatter_kernel made (listed references page_cnt,
// first list position page_first):
//  - a page is eligible when every reference to it is selected (selected
//    references == reference count), and is planned once, at its first
//    selected position;
//  - mirror mode: eligible pages whose host copy is stale form the copy
//    list, and are marked current (full pages only) for the copy about to be
//    issued;
//  - per selected key: its slot (plan position, or page id in mirror mode),
//    -1 when its page is not eligible.
// page_cnt / page_first are restored to 0 / ~0 before returning.
__global__ void __launch_bounds__(1024) plan_kernel(const Work w, uint32_t mirror, const SelectOut out)
{
    __shared__ uint32_t wsum[33];
    pdl_wait();                 // the list and page counts come from the selection
    pdl_trigger();
    const uint32_t n = *w.sel_count;
    if (n <= 4 * blockDim.x) {
        // one pass with every entry's loads in registers: 4 consecutive
        // entries per thread
        const uint32_t i0 = 4 * threadIdx.x;
        int32_t p[4];
        uint32_t cnt[4], ref[4], lead[4], dirty[4], nl = 0, nd = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            p[q] = i0 + q < n ? w.sel_pages[i0 + q] : -1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            cnt[q] = ref[q] = lead[q] = dirty[q] = 0;
            if (p[q] >= 0) {
                cnt[q] = w.page_cnt[p[q]];
                ref[q] = w.dev_refcnt[p[q]];
                lead[q] = (cnt[q] == ref[q] && w.page_first[p[q]] == i0 + q) ? 1u : 0u;
                dirty[q] = (lead[q] && mirror && !w.page_clean[p[q]]) ? 1u : 0u;
            }
            nl += lead[q];
            nd += dirty[q];
        }
        uint32_t tot;
        const uint32_t ex = block_scan_1024(nl | (nd << 16), wsum, &tot);
        uint32_t pos = ex & 0xffffu, cpos = ex >> 16;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (lead[q]) {
                w.plan_pages[pos] = p[q];
                w.page_pos[p[q]] = static_cast<int32_t>(pos);
                ++pos;
            }
            if (dirty[q]) {
                w.readback[4 + cpos] = static_cast<uint32_t>(p[q]);
                w.page_clean[p[q]] = w.sel_full[i0 + q];
                ++cpos;
            }
        }
        __syncthreads();        // page_pos of every leader is written
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t i = i0 + q;
            if (i < n) {
                const int32_t v = (p[q] >= 0 && cnt[q] == ref[q]) ? (mirror ? p[q] : w.page_pos[p[q]]) : -1;
                w.plan_slot[i] = v;
                if (out.slots && i < out.ids_cap)
                    out.slots[i] = v;
            }
            if (p[q] >= 0) {    // every read of the counts was before the scan's barriers
                w.page_cnt[p[q]] = 0;
                w.page_first[p[q]] = 0xffffffffu;
            }
        }
        if (threadIdx.x == 0) {
            w.readback[0] = n;
            w.readback[1] = tot & 0xffffu;
            w.readback[2] = tot >> 16;
            w.readback[3] = 0;
            if (out.count_host) {
                out.count_host[0] = n;
                out.count_host[1] = tot & 0xffffu;
                out.count_host[2] = tot >> 16;
                out.count_host[3] = 0;
            }
        }
        return;
    }
    // leaders in list order: 4 consecutive entries per thread per tile; one
    // block scan of the packed counts (leaders low 16 bits, stale pages high:
    // at most 4,096 of each per tile)
    uint32_t npages = 0, ncopy = 0;
    for (uint32_t t0 = 0; t0 < n; t0 += 4 * blockDim.x) {
        const uint32_t i0 = t0 + 4 * threadIdx.x;
        int32_t p[4];
        uint32_t lead[4], dirty[4], nl = 0, nd = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t i = i0 + q;
            lead[q] = dirty[q] = 0;
            p[q] = 0;
            if (i < n) {
                p[q] = w.sel_pages[i];
                lead[q] = (w.page_cnt[p[q]] == w.dev_refcnt[p[q]] && w.page_first[p[q]] == i) ? 1u : 0u;
                dirty[q] = (lead[q] && mirror && !w.page_clean[p[q]]) ? 1u : 0u;
            }
            nl += lead[q];
            nd += dirty[q];
        }
        uint32_t tot;
        const uint32_t ex = block_scan_1024(nl | (nd << 16), wsum, &tot);
        uint32_t pos = npages + (ex & 0xffffu), cpos = ncopy + (ex >> 16);
        npages += tot & 0xffffu;
        ncopy += tot >> 16;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (lead[q]) {
                w.plan_pages[pos] = p[q];
                w.page_pos[p[q]] = static_cast<int32_t>(pos);
                ++pos;
            }
            if (dirty[q]) {
                w.readback[4 + cpos] = static_cast<uint32_t>(p[q]);
                w.page_clean[p[q]] = w.sel_full[i0 + q];
                ++cpos;
            }
        }
    }
    __syncthreads();
    // slots: 8 entries per thread per pass, every load of a pass issued
    // before its stores
    constexpr int R = 8;
    for (uint32_t t0 = 0; t0 < n; t0 += R * blockDim.x) {
        int32_t p[R];
        uint32_t cnt[R], ref[R];
        int32_t pos[R];
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const uint32_t i = t0 + q * blockDim.x + threadIdx.x;
            p[q] = i < n ? w.sel_pages[i] : -1;
        }
#pragma unroll
        for (int q = 0; q < R; ++q) {
            cnt[q] = ref[q] = 0;
            pos[q] = -1;
            if (p[q] >= 0) {
                cnt[q] = w.page_cnt[p[q]];
                ref[q] = w.dev_refcnt[p[q]];
                pos[q] = mirror ? p[q] : w.page_pos[p[q]];
            }
        }
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const uint32_t i = t0 + q * blockDim.x + threadIdx.x;
            if (i < n) {
                const int32_t v = (p[q] >= 0 && cnt[q] == ref[q]) ? pos[q] : -1;
                w.plan_slot[i] = v;
                if (out.slots && i < out.ids_cap)
                    out.slots[i] = v;
            }
        }
    }
    __syncthreads();
    // page_cnt / page_first back to 0 / ~0 for the next plan
    for (uint32_t t0 = 0; t0 < n; t0 += R * blockDim.x) {
        int32_t p[R];
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const uint32_t i = t0 + q * blockDim.x + threadIdx.x;
            p[q] = i < n ? w.sel_pages[i] : -1;
        }
#pragma unroll
        for (int q = 0; q < R; ++q)
            if (p[q] >= 0) {
                w.page_cnt[p[q]] = 0;
                w.page_first[p[q]] = 0xffffffffu;
            }
    }
    if (threadIdx.x == 0) {
        w.readback[0] = n;
        w.readback[1] = npages;
        w.readback[2] = ncopy;
        w.readback[3] = 0;
        if (out.count_host) {
            out.count_host[0] = n;
            out.count_host[1] = npages;
            out.count_host[2] = ncopy;
            out.count_host[3] = 0;
        }
    }
}

// ------------------------------------------------------------------- gather
// grid.x = pages, grid.y = parts of a page; 16-byte vector copies.
__global__ void __launch_bounds__(256)
    gather_kernel(const uint4 *pool, const int32_t *pages, uint4 *staging, uint64_t page_vec)
{
    const int32_t page = pages[blockIdx.x];
    const uint4 *src = pool + static_cast<uint64_t>(page) * page_vec;
    uint4 *dst = staging + static_cast<uint64_t>(blockIdx.x) * page_vec;
    const uint64_t per = (page_vec + gridDim.y - 1) / gridDim.y;
    const uint64_t a = blockIdx.y * per;
    const uint64_t e = min(page_vec, a + per);
    for (uint64_t i = a + threadIdx.x; i < e; i += blockDim.x)
        dst[i] = __ldcs(src + i);
}

// The plan's stale pages (plan[2] of them, page ids from plan + 4) straight
// into the host mirror through its device mapping: pool page p to host page
// p.  Every CTA takes its slice of every page (no division per element); an
// id outside the pool is flagged and skipped.
//
// Completion goes to the host through pinned memory, not a stream event
// (an event between this kernel and the next step's first kernel would make
// that a plain launch): hdr[0..3] receive the counts plan[0..2] and 0, then
// hdr[4] the call's sequence number, once every copy of the call is visible
// to the host.  The copying threads fence at system scope and their CTAs
// count themselves on plan[3] (0 from the plan kernel); the CTA that
// arrives last publishes.  With nothing to copy CTA 0 publishes at once.
__global__ void __launch_bounds__(256)
    mirror_copy_kernel(const uint4 *pool, uint32_t *plan, uint4 *host, uint64_t page_vec,
                       uint32_t pool_blocks, uint32_t *err, uint32_t *err_info, uint32_t *hdr, uint32_t seq)
{
    pdl_wait();                 // the copy list comes from the plan kernel
    pdl_trigger();
    const uint32_t n = plan[2];
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
    const uint64_t i0 = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (uint32_t k = 0; k < n; ++k) {
        const uint32_t p = plan[4 + k];
        if (p >= pool_blocks) {
            if (i0 == 0) {
                atomicOr(err, kErrBadPage);
                atomicCAS(err_info, 0u, p | 0x80000000u);
            }
            continue;
        }
        const uint4 *src = pool + p * page_vec;
        uint4 *dst = host + p * page_vec;
        uint64_t i = i0;
        for (; i + 3 * stride < page_vec; i += 4 * stride) {
            const uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride);
            const uint4 c = __ldcs(src + i + 2 * stride), d = __ldcs(src + i + 3 * stride);
            dst[i] = a;
            dst[i + stride] = b;
            dst[i + 2 * stride] = c;
            dst[i + 3 * stride] = d;
        }
        for (; i < page_vec; i += stride)
            dst[i] = __ldcs(src + i);
    }
    if (!hdr)
        return;                 // uniform over the grid
    if (n)
        __threadfence_system(); // this thread's host writes, before its CTA arrives
    __syncthreads();
    if (threadIdx.x == 0) {
        bool last = blockIdx.x == 0;
        if (n) {
            __threadfence_system();
            last = atomicAdd(plan + 3, 1u) == gridDim.x - 1;
        }
        if (last) {
            if (n)
                __threadfence_system(); // every CTA's copies before the counts and the tag
            volatile uint32_t *h = hdr;
            h[0] = plan[0];
            h[1] = plan[1];
            h[2] = n;
            h[3] = 0;
            __threadfence_system();
            h[4] = seq;
        }
    }
}

// staging page i -> pool page pages[i] (re-admission); grid.y = parts of a page
__global__ void __launch_bounds__(256)
    scatter_kernel(const uint4 *staging, const int32_t *pages, uint4 *pool, uint64_t page_vec)
{
    const int32_t page = pages[blockIdx.x];
    const uint4 *src = staging + static_cast<uint64_t>(blockIdx.x) * page_vec;
    uint4 *dst = pool + static_cast<uint64_t>(page) * page_vec;
    const uint64_t per = (page_vec + gridDim.y - 1) / gridDim.y;
    const uint64_t a = blockIdx.y * per;
    const uint64_t e = min(page_vec, a + per);
    for (uint64_t i = a + threadIdx.x; i < e; i += blockDim.x)
        dst[i] = __ldcs(src + i);
}

// The decode set from the kernel's parameters into device memory.
struct SetBlob {
    uint4 v[kSetInlineBytes / 16];
};

__global__ void __launch_bounds__(256) set_kernel(const __grid_constant__ SetBlob b, uint32_t nvec, uint4 *dst)
{
    pdl_trigger();
    pdl_wait();                 // earlier kernels of the stream may still read the old set
    for (uint32_t i = threadIdx.x; i < nvec; i += blockDim.x)
        dst[i] = b.v[i];
}

__global__ void patch_kernel(const Geo g, int32_t *table, kvs_record *recs, uint8_t *page_clean,
                             const Patch *p, uint32_t n)
{
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n)
        return;
    const Patch q = p[i];
    const size_t idx = static_cast<size_t>(q.slot) * g.mb + q.block;
    table[idx] = q.page;
    if (q.page >= 0 && (q.what & kPatchPageWritten))
        page_clean[q.page] = 0;          // page bytes were rewritten (readmit)
    if (q.what & kPatchRecord)
        recs[idx] = q.rec;
}

__global__ void copy_mass_kernel(const Geo g, const Work w, const float *src, float *mass)
{
    const DSet *ds = w.dset;
    const uint32_t ci = blockIdx.y;
    const DSeq sq = ds->seq[ci];
    for (uint32_t b = blockIdx.x * blockDim.x + threadIdx.x; b < sq.nb; b += gridDim.x * blockDim.x)
        mass[static_cast<size_t>(sq.slot) * g.mb + b] = src[static_cast<size_t>(ci) * g.mb + b];
}

}  // namespace

cudaError_t launch_append(const Geo &g, const AppendArgs &a, cudaStream_t s)
{
    const uint32_t vec_per_row = g.d * (g.fp8 ? 1 : 2) / 16;   // 16-byte page vectors per row
    // rows cover every slot from p0 to the end of the last touched block
    const uint64_t slots = static_cast<uint64_t>(a.first_blk + a.nblk) * kBlockTokens - a.p0;
    const uint64_t rows = slots * g.L * 2 * g.Hkv;
    const uint64_t threads = rows * vec_per_row + a.nblk;   // nblk >= new blocks
    const uint32_t bs = 256;
    const uint64_t grid = (threads + bs - 1) / bs;
    if (grid > 0x7fffffffull)
        return cudaErrorInvalidValue;
    append_kernel<<<static_cast<uint32_t>(grid), bs, 0, s>>>(g, a, rows, vec_per_row);
    return cudaGetLastError();
}

cudaError_t launch_append_step(const Geo &g, const uint16_t *k, const uint16_t *v, uint16_t *pool,
                               int32_t *table, kvs_record *records, uint8_t *page_clean,
                               const StepAppend *sa_dev, const StepAppend *sa_host, uint32_t nseq,
                               uint32_t rows_total, uint64_t t_create, cudaStream_t s)
{
    const uint32_t vec_per_row = g.d * (g.fp8 ? 1 : 2) / 16;   // 16-byte page vectors per row
    const uint64_t threads = static_cast<uint64_t>(rows_total) * vec_per_row + nseq;
    const uint32_t bs = 256;
    StepAppendInline inl{};
    if (!sa_dev) {
        if (nseq > kStepInline)
            return cudaErrorInvalidValue;
        for (uint32_t i = 0; i < nseq; ++i)
            inl.e[i] = sa_host[i];
    }
    return launch_pdl(append_step_kernel, dim3(static_cast<uint32_t>((threads + bs - 1) / bs)), dim3(bs), 0, s,
                      g, k, v, pool, table, records, page_clean, sa_dev, inl, nseq, rows_total, vec_per_row,
                      t_create);
}

cudaError_t launch_score(const Geo &g, const Work &w, kvs_record *rec, const float *mass,
                         double alpha, uint32_t W, double wR, double wE, double wN, double lo,
                         double hi, uint32_t nb_total, cudaStream_t s)
{
    ScoreArgs sa{alpha, wR, wE, wN, lo, hi, W};
    return launch_pdl(score_kernel, dim3((nb_total + 127) / 128), dim3(128), 0, s, g, w, rec, mass, sa, nb_total);
}

cudaError_t launch_radix_select(const Geo &g, const Work &w, const kvs_record *rec,
                                uint32_t nb_total, uint32_t k, int mode, double alpha, cudaStream_t s)
{
    return launch_pdl(radix_select_kernel, dim3(1), dim3(1024), 0, s, g, w, rec, nb_total, k, mode, alpha);
}

cudaError_t launch_select(const Geo &g, const Work &w, const kvs_record *rec, const int32_t *table,
                          int mode, double alpha, uint32_t nb_total, bool count_pages, const SelectOut &out,
                          cudaStream_t s)
{
    const uint32_t ntiles = (nb_total + kSelTile - 1) / kSelTile;
    if (ntiles > 1) {           // one tile counts itself in the scatter kernel
        cudaError_t e = launch_pdl(select_count_kernel, dim3(ntiles), dim3(kSelThreads), 0, s, g, w, rec, mode,
                                   alpha, nb_total);
        if (e != cudaSuccess)
            return e;
    }
    return launch_pdl(select_scatter_kernel, dim3(ntiles), dim3(kSelThreads), 0, s, g, w, rec, table, mode, alpha,
                      nb_total, ntiles, count_pages ? 1u : 0u, out);
}

bool select_plan_fits(uint32_t nb_total) { return nb_total <= kSelOneTile; }

cudaError_t launch_select_plan(const Geo &g, const Work &w, const kvs_record *rec, const int32_t *table, int mode,
                               double alpha, uint32_t nb_total, uint32_t mirror, const SelectOut &out,
                               cudaStream_t s)
{
    if (nb_total > kSelOneTile)
        return cudaErrorInvalidValue;
    return launch_pdl(select_plan_kernel, dim3(1), dim3(kSelOneTile), 0, s, g, w, rec, table, mode, alpha,
                      nb_total, mirror, out);
}

uint32_t select_launches(uint32_t nb_total)
{
    return nb_total > static_cast<uint32_t>(kSelTile) ? 2u : 1u;
}

cudaError_t launch_prefetch_plan(const PrefCand *cand, uint32_t n, uint32_t k, uint64_t *keys,
                                 uint64_t *out_key, uint32_t *out_idx, cudaStream_t s)
{
    if (k == 0 || k > KVS_PREFETCH_MAX || k > n)
        return cudaErrorInvalidValue;
    const int smem = KVS_PREFETCH_MAX * (sizeof(uint64_t) + sizeof(uint32_t));
    cudaError_t e = cudaFuncSetAttribute(prefetch_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return e;
    prefetch_plan_kernel<<<1, 1024, smem, s>>>(cand, n, k, keys, out_key, out_idx);
    return cudaGetLastError();
}

cudaError_t launch_gather(const Geo &g, const uint16_t *pool, const int32_t *pages, uint32_t npages,
                          uint8_t *staging, cudaStream_t s)
{
    const uint64_t page_vec = g.page_bytes / 16;
    const uint32_t parts = static_cast<uint32_t>(std::max<uint64_t>(1, std::min<uint64_t>(64, page_vec / 4096)));
    gather_kernel<<<dim3(npages, parts), 256, 0, s>>>(reinterpret_cast<const uint4 *>(pool), pages,
                                                     reinterpret_cast<uint4 *>(staging), page_vec);
    return cudaGetLastError();
}

cudaError_t launch_mirror_copy(const Geo &g, const Work &w, const uint16_t *pool, void *host_dev,
                               uint32_t pool_blocks, int grid, uint32_t *hdr_dev, uint32_t seq, cudaStream_t s)
{
    return launch_pdl(mirror_copy_kernel, dim3(grid), dim3(256), 0, s, reinterpret_cast<const uint4 *>(pool),
                      w.readback, reinterpret_cast<uint4 *>(host_dev), static_cast<uint64_t>(g.page_bytes / 16),
                      pool_blocks, w.err, w.err_info, hdr_dev, seq);
}

cudaError_t launch_scatter(const Geo &g, const uint8_t *staging, const int32_t *pages, uint32_t npages,
                           uint16_t *pool, cudaStream_t s)
{
    const uint64_t page_vec = g.page_bytes / 16;
    const uint32_t parts = static_cast<uint32_t>(std::max<uint64_t>(1, std::min<uint64_t>(64, page_vec / 4096)));
    scatter_kernel<<<dim3(npages, parts), 256, 0, s>>>(reinterpret_cast<const uint4 *>(staging), pages,
                                                      reinterpret_cast<uint4 *>(pool), page_vec);
    return cudaGetLastError();
}

cudaError_t launch_set(const void *src, size_t bytes, void *dst, cudaStream_t s)
{
    if (bytes > kSetInlineBytes)
        return cudaErrorInvalidValue;
    SetBlob b;
    std::memset(&b, 0, sizeof b);
    std::memcpy(&b, src, bytes);
    const uint32_t nvec = static_cast<uint32_t>((bytes + 15) / 16);
    return launch_pdl(set_kernel, dim3(1), dim3(256), 0, s, b, nvec, static_cast<uint4 *>(dst));
}

cudaError_t launch_patch(const Geo &g, int32_t *table, kvs_record *rec, uint8_t *page_clean,
                         const Patch *p, uint32_t n, cudaStream_t s)
{
    patch_kernel<<<(n + 127) / 128, 128, 0, s>>>(g, table, rec, page_clean, p, n);
    return cudaGetLastError();
}

cudaError_t launch_plan(const Work &w, uint32_t mirror, const SelectOut &out, cudaStream_t s)
{
    return launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, s, w, mirror, out);
}

cudaError_t launch_copy_mass(const Geo &g, const Work &w, const float *src, float *mass,
                             uint32_t nseq, cudaStream_t s)
{
    copy_mass_kernel<<<dim3(std::max<uint32_t>(1, (g.mb + 255) / 256), nseq), 256, 0, s>>>(g, w, src, mass);
    return cudaGetLastError();
}

}  // namespace kvs
