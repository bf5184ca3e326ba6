// KIVI-style 2-bit KV (sm_103a): group quantisation and the decode kernel
// over group pages.
//
// Source: "Fitting a Million Tokens", s.02 "Quantize the cache" (KIVI): keys
// per channel over groups of 32 tokens -- two 16-token blocks, so the group
// is dequantised at block granularity inside the attention kernel -- values
// per token over groups of 32 channels, asymmetric 2-bit codes with an fp16
// scale and zero per group, the newest ~128 tokens kept unquantised.
//
//   kivi_compress_kernel -- one CTA of 128 threads per (group, layer, KV
//                           head): reads the group's 32 bf16 tokens from its
//                           two pages, quantises K per channel and V per
//                           (token, 32-channel group) in fp32 with explicit
//                           rounding, and writes the 3072-byte tile in the
//                           layout the decode warps read.
//   decode_kivi_kernel   -- persistent, independent warps as in the page
//                           decode: each claims (sequence, layer, KV head,
//                           chunk of groups) items and streams 3 KiB group
//                           tiles through a bulk-copy ring.  Codes become
//                           f16 pairs code/2 by the FP4 (e2m1) pair
//                           conversion (exact).  Keys: fp16(code*s + z) by one
//                           f16 fused multiply-add per pair, (code/2)(2s) + z
//                           -- the quantiser's dequantised value, one
//                           rounding -- into the S MMAs.  Values are s_t*code +
//                           z_t per token and channel group, and never formed:
//                           O^T += (codes/2) . (2 s_t P^T) per m-tile, and the
//                           zero term, one value per (channel group, head), by
//                           one MMA per block whose rows are the four channel
//                           groups, added to O at the end of the item.  It
//                           writes the
//                           same split-K partials and per-block log2-sum-exps
//                           as the page decode.
//
// Tile layout (per (layer, KV head) of a group page; lane = 4g + t).  A code
// word holds operand pairs as the 2-bit low fields of a byte's two nibbles:
// byte k of word w carries register k of step 2w (fields 0-1 and 4-5, first
// element low) and register k of step 2w + 1 (fields 2-3 and 6-7), so
// (w & 0x33333333) and ((w >> 2) & 0x33333333) are each four FP4 pairs.
// Scales are held doubled (2s, exact in fp16), the factor the code/2 operands
// need.
//   [0, 1024)    K codes [block j][lane][word w]: step s = k-step s (16
//                channels), register r: token 16j + g + 8(r%2), channels
//                (c, c+8) for r < 2 and (c+1, c+9) for r >= 2,
//                c = 32t + 16(s/4) + 2(s%4).
//   [1024, 2048) V codes [block j][lane][word w]: step s = m-tile s,
//                register r: channel 16s + g + 8(r%2), tokens 16j + 2t +
//                8(r/2) and the next one.
//   [2048, 2560) K (2 x scale pair, zero pair) [h][ip][t][i = 2ip, 2ip+1]:
//                channels 32t + 16h + i (low half) and + 8 (high half); the
//                four t of one (h, ip) are 64 contiguous bytes, so the 16-byte
//                loads of the lanes t = 0..3 fall in different banks.
//   [2560, 2816) V 2 x scale pairs [block j][token pair p][channel group c]:
//                tokens 16j + 2p (low) and 16j + 2p + 1 (high);
//   [2816, 3072) V zero pairs, the same order.
#include <cuda_fp16.h>

#include "kvs_internal.h"
#include "kvs_pdl.cuh"
#include "kvs_ptx.h"

namespace kvs {
namespace {

using namespace ptx;

constexpr uint32_t kTile = KVS_KIVI_TILE_BYTES;
constexpr int kKRing = 6;           // group tiles in flight per warp
constexpr int kKWarps = 4;          // warps per CTA
constexpr int kKMinCtas = 3;        // CTAs per SM (12 warps: dequantisation is ALU work)
constexpr uint32_t kKClaimLead = 2; // groups between claiming an item and needing its tiles
constexpr int kKD = 128;            // head dimension of the scheme

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__device__ __forceinline__ uint16_t h_bits(__half h) { return __half_as_ushort(h); }

// ------------------------------------------------------------------ compress
__global__ void __launch_bounds__(128)
    kivi_compress_kernel(const Geo g, const KiviJob *jobs, const uint8_t *pool, uint8_t *gpool,
                         int32_t *table)
{
    __shared__ uint8_t kc[32][kKD];
    __shared__ uint8_t vc[32][kKD];
    __shared__ uint16_t sk[kKD], zk[kKD];
    __shared__ uint16_t sv[32][4], zv[32][4];
    __shared__ uint32_t tile[kTile / 4];
    const uint32_t LH = g.L * g.Hkv;
    const KiviJob job = jobs[blockIdx.x / LH];
    const uint32_t lh = blockIdx.x % LH;
    const uint32_t l = lh / g.Hkv, h = lh % g.Hkv;
    const uint32_t tid = threadIdx.x;
    // token t of the group: page of block t / 16, slot t % 16
    auto row = [&](uint32_t t, uint32_t kv) -> const uint16_t * {
        const int32_t page = t < 16 ? job.page0 : job.page1;
        return reinterpret_cast<const uint16_t *>(
            pool + static_cast<uint64_t>(page) * g.page_bytes +
            ((((static_cast<uint64_t>(l) * 2 + kv) * g.Hkv + h) * kBlockTokens + (t & 15)) * kKD) * 2);
    };
    // keys: thread = channel, over the 32 tokens
    {
        float x[32];
        float mn = INFINITY, mx = -INFINITY;
#pragma unroll
        for (uint32_t t = 0; t < 32; ++t) {
            x[t] = bf16f(row(t, 0)[tid]);
            mn = fminf(mn, x[t]);
            mx = fmaxf(mx, x[t]);
        }
        const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 3.0f));
        const __half z16 = __float2half_rn(mn);
        const float sf = __half2float(s16), zf = __half2float(z16);
#pragma unroll
        for (uint32_t t = 0; t < 32; ++t) {
            int c = 0;
            if (sf > 0.f)
                c = min(max(__float2int_rn(__fdiv_rn(__fsub_rn(x[t], zf), sf)), 0), 3);
            kc[t][tid] = static_cast<uint8_t>(c);
        }
        sk[tid] = h_bits(__hadd(s16, s16));    // the tile holds 2s (exact)
        zk[tid] = h_bits(z16);
    }
    // values: thread = (token, channel group), over 32 channels
    {
        const uint32_t t = tid >> 2, cg = tid & 3;
        const uint4 *src = reinterpret_cast<const uint4 *>(row(t, 1) + 32 * cg);
        float x[32];
        float mn = INFINITY, mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = src[q];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[8 * q + 2 * e] = __uint_as_float(w[e] << 16);
                x[8 * q + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
            }
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            mn = fminf(mn, x[e]);
            mx = fmaxf(mx, x[e]);
        }
        const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 3.0f));
        const __half z16 = __float2half_rn(mn);
        const float sf = __half2float(s16), zf = __half2float(z16);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            int c = 0;
            if (sf > 0.f)
                c = min(max(__float2int_rn(__fdiv_rn(__fsub_rn(x[e], zf), sf)), 0), 3);
            vc[t][32 * cg + e] = static_cast<uint8_t>(c);
        }
        sv[t][cg] = h_bits(__hadd(s16, s16));
        zv[t][cg] = h_bits(z16);
    }
    __syncthreads();
    // code words: 256 K words and 256 V words, index (j * 32 + lane) * 4 + w;
    // byte k of word w: register k of step 2w (fields 0-1 and 4-5) and of
    // step 2w + 1 (fields 2-3 and 6-7), first element in the low field
    for (uint32_t wi = tid; wi < 256; wi += blockDim.x) {
        const uint32_t j = wi >> 7, lane = (wi >> 2) & 31, w = wi & 3;
        const uint32_t gq = lane >> 2, tq = lane & 3;
        uint32_t kw = 0, vw = 0;
#pragma unroll
        for (uint32_t k = 0; k < 4; ++k) {
#pragma unroll
            for (uint32_t half = 0; half < 2; ++half) {
                const uint32_t st = 2 * w + half, lo = 8 * k + 2 * half, hi = lo + 4;
                // K step st: token 16j + g + 8(k % 2), channels (c, c + 8)
                const uint32_t tok = 16 * j + gq + 8 * (k & 1);
                const uint32_t c = 32 * tq + 16 * (st >> 2) + 2 * (st & 3) + (k >> 1);
                kw |= (static_cast<uint32_t>(kc[tok][c]) << lo) | (static_cast<uint32_t>(kc[tok][c + 8]) << hi);
                // V m-tile st: channel 16 st + g + 8(k % 2), tokens t0 and t0 + 1
                const uint32_t ch = 16 * st + gq + 8 * (k & 1);
                const uint32_t t0 = 16 * j + 2 * tq + 8 * (k >> 1);
                vw |= (static_cast<uint32_t>(vc[t0][ch]) << lo) | (static_cast<uint32_t>(vc[t0 + 1][ch]) << hi);
            }
        }
        tile[wi] = kw;
        tile[256 + wi] = vw;
    }
    {
        // K meta: (((h * 4 + ip) * 4 + t) * 2 + di) * 2 + which, i = 2ip + di
        const uint32_t which = tid & 1, di = (tid >> 1) & 1, tq = (tid >> 2) & 3, ip = (tid >> 4) & 3,
                       hh = tid >> 6;
        const uint32_t ch = 32 * tq + 16 * hh + 2 * ip + di;
        const uint16_t *src = which ? zk : sk;
        tile[512 + tid] = static_cast<uint32_t>(src[ch]) | (static_cast<uint32_t>(src[ch + 8]) << 16);
        // V meta: the scales, then the zeros, each [j][p][c]: vwhich * 64 +
        // (j * 8 + p) * 4 + c
        const uint32_t vwhich = tid >> 6, cg = tid & 3, p = (tid >> 2) & 7, j = (tid >> 5) & 1;
        const uint32_t tok = 16 * j + 2 * p;
        const uint16_t(*vsrc)[4] = vwhich ? zv : sv;
        tile[640 + tid] = static_cast<uint32_t>(vsrc[tok][cg]) | (static_cast<uint32_t>(vsrc[tok + 1][cg]) << 16);
    }
    __syncthreads();
    uint32_t *dst = reinterpret_cast<uint32_t *>(gpool + static_cast<uint64_t>(job.gpage) * g.group_page_bytes +
                                                 static_cast<uint64_t>(lh) * kTile);
    for (uint32_t i = tid; i < kTile / 4; i += blockDim.x)
        dst[i] = tile[i];
    if (lh == 0 && tid == 0) {
        int32_t *trow = table + static_cast<size_t>(job.slot) * g.mb;
        trow[2 * job.group] = KVS_TABLE_GROUP(job.gpage);
        trow[2 * job.group + 1] = KVS_TABLE_GROUP(job.gpage);
    }
}

// -------------------------------------------------------------------- decode
struct KArgs {
    Geo g;
    Work w;
    const uint16_t *q;
    const int32_t *table;
    const uint8_t *gpool;
    uint32_t n_items;
};

struct KItem {
    uint32_t valid;
    uint32_t ci, l, kvh;
    uint32_t g0;        // first group
    uint32_t ng;        // groups in the item
    uint32_t part, lse0;
};

struct KPrep {
    KItem it;
    int32_t gp[2];      // group pages: lane j holds groups j and j + 32
};

__device__ __forceinline__ KPrep prepare_kitem(const KArgs &a, uint32_t id, uint32_t lane)
{
    KPrep p;
    p.it.valid = 0;
    p.it.ng = 0;
    if (id >= a.n_items)
        return p;
    const DSet *ds = a.w.dset;
    const Geo &g = a.g;
    const uint32_t ci = find_seq(&ds->seq[0].item_off_q, sizeof(DSeq) / 4, ds->nseq, id);
    const DSeq &sq = ds->seq[ci];
    // chunk-major, KV head fastest, as the page items: large chunks first,
    // the short ones last (all chunk sizes even: whole groups)
    uint32_t local = id - sq.item_off_q;
    const uint32_t kvh = local % g.Hkv;
    local /= g.Hkv;
    const uint32_t l = local % g.L;
    const uint32_t chunk = local / g.L;
    const uint32_t b0 = chunk < sq.nbig_q ? chunk * ds->chunk
                                          : sq.nbig_q * ds->chunk + (chunk - sq.nbig_q) * ds->chunk_q_small;
    const uint32_t size = chunk < sq.nbig_q ? ds->chunk : ds->chunk_q_small;
    const uint32_t nblk = min(size, sq.qb - b0);
    p.it.valid = 1;
    p.it.ci = ci;
    p.it.l = l;
    p.it.kvh = kvh;
    p.it.g0 = b0 / 2;
    p.it.ng = nblk / 2;
    p.it.part = sq.part_off + (l * g.Hkv + kvh) * sq.nchunk + chunk;
    p.it.lse0 = sq.blk_off + b0;
    const int32_t *trow = a.table + static_cast<size_t>(sq.slot) * g.mb + b0;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint32_t j = lane + 32 * q;
        int32_t gp = 0;
        if (j < p.it.ng) {
            const int32_t v = __ldg(trow + 2 * j);
            gp = -2 - v;
            if (v > -2 || gp >= static_cast<int32_t>(g.kivi_groups)) {
                atomicOr(a.w.err, kErrBadPage);
                atomicCAS(a.w.err_info, 0u, static_cast<uint32_t>(v) | 0x80000000u);
                gp = 0;
            }
        }
        p.gp[q] = gp;
    }
    return p;
}

struct KRing {
    uint32_t inflight, st_issue, st_cons, ph_cons;
};

// Issues the next group tile of the warp's stream (items cur, then nxt).
__device__ __forceinline__ bool kissue_next(const KArgs &a, const KPrep &cur, const KPrep &nxt, bool have_nxt,
                                            bool &c_in_nxt, uint32_t &c_grp, KRing &rg, uint32_t ring_u32,
                                            uint64_t *bars, uint32_t lane)
{
    if (!c_in_nxt && c_grp >= cur.it.ng) {
        if (!have_nxt || !nxt.it.valid)
            return false;
        c_in_nxt = true;
        c_grp = 0;
    }
    if (c_in_nxt && c_grp >= nxt.it.ng)
        return false;
    const KPrep &pp = c_in_nxt ? nxt : cur;
    const int32_t gsel = c_grp < 32 ? pp.gp[0] : pp.gp[1];
    const int32_t gp = __shfl_sync(0xffffffffu, gsel, c_grp & 31);
    if (lane == 0) {
        const uint32_t st = rg.st_issue;
        const uint32_t bar = smem_u32(&bars[st]);
        mbar_expect_tx(bar, kTile);
        const uint8_t *src = a.gpool + static_cast<uint64_t>(gp) * a.g.group_page_bytes +
                             (static_cast<uint64_t>(pp.it.l) * a.g.Hkv + pp.it.kvh) * kTile;
        bulk_load(ring_u32 + st * kTile, src, kTile, bar, l2_evict_first());
    }
    ++c_grp;
    ++rg.inflight;
    rg.st_issue = rg.st_issue + 1 == kKRing ? 0 : rg.st_issue + 1;
    return true;
}

// The four bytes of a masked code word (each byte two 2-bit codes in the low
// fields of its nibbles) as four f16 pairs code/2: a 2-bit field in the low
// bits of an FP4 (e2m1) nibble is the value code/2 exactly (0, 0.5, 1, 1.5),
// and the hardware conversion takes a byte of two nibbles to an f16 pair
// (low nibble to the low half).
__device__ __forceinline__ void e2m1x4(uint32_t m, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
        : "r"(m));
}

__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b)
{
    const __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
    return *reinterpret_cast<const uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c)
{
    const __half2 r = __hfma2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b),
                              *reinterpret_cast<const __half2 *>(&c));
    return *reinterpret_cast<const uint32_t *>(&r);
}

constexpr uint32_t kCodeMask = 0x33333333u;    // the low fields of both nibbles of every byte

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t lo_bits, uint32_t hi_bits)
{
    return pack_f16(__uint_as_float(lo_bits << 16), __uint_as_float(hi_bits << 16));
}

__global__ void __launch_bounds__(32 * kKWarps, kKMinCtas) decode_kivi_kernel(const KArgs a)
{
    extern __shared__ __align__(1024) uint8_t ksm_raw[];
    __shared__ __align__(8) uint64_t bars[kKWarps][kKRing];
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(ksm_raw) + 127) & ~uintptr_t(127));
    const uint32_t ring_u32 = smem_u32(smem + warp * kKRing * kTile);
    if (lane == 0) {
        for (int s = 0; s < kKRing; ++s)
            mbar_init(smem_u32(&bars[warp][s]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
    // a programmatic dependent, as the page decode: nothing in global memory
    // before the kernel ahead has completed; then the next kernel (the page
    // decode of the residual, or the combine) may place its CTAs
    pdl_wait();
    pdl_trigger();

    const Geo &g = a.g;
    const uint32_t G = g.G;
    const uint32_t gq = lane >> 2, tq = lane & 3;
    const uint32_t h0 = 2 * tq, h1 = 2 * tq + 1;
    const float scale_log2 = rsqrtf(static_cast<float>(kKD)) * kLog2e;
    const uint32_t nb_total = a.w.dset->nb_total;
    uint32_t *counter = a.w.counter + 1;

    // one item claimed at a time, shortly before the ring needs its first
    // tile (as in the page decode kernel)
    auto claim = [&]() -> uint32_t {
        uint32_t id = 0;
        if (lane == 0)
            id = atomicAdd(counter, 1u);
        return __shfl_sync(0xffffffffu, id, 0);
    };
    KPrep cur = prepare_kitem(a, claim(), lane);
    KPrep nxt;
    nxt.it.valid = 0;
    nxt.it.ng = 0;
    bool have_nxt = false;
    KRing rg{0, 0, 0, 0};
    bool c_in_nxt = false;
    uint32_t c_grp = 0;
    if (cur.it.valid)
        while (rg.inflight < kKRing &&
               kissue_next(a, cur, nxt, have_nxt, c_in_nxt, c_grp, rg, ring_u32, bars[warp], lane)) {
        }

    while (cur.it.valid) {
        const KItem it = cur.it;
        const uint32_t kvh = it.kvh;
        const uint32_t claim_at = it.ng > kKRing + kKClaimLead ? it.ng - kKRing - kKClaimLead : 0;
        // query fragments for the lane's head gq: channels 32tq + 16(ks/4) +
        // {i0, i0+8} (b0) and {i0+1, i0+9} (b1), i0 = 2(ks%4) -- the pairs
        // the K code words hold
        uint32_t qf[8][2];
        {
            const bool valid = gq < G;
            const uint16_t *qh = a.q + ((static_cast<size_t>(it.ci) * g.L + it.l) * g.Hq + kvh * G +
                                        (valid ? gq : 0)) * kKD + 32 * tq;
            uint32_t qw[16];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 x = valid ? __ldg(reinterpret_cast<const uint4 *>(qh) + v) : make_uint4(0, 0, 0, 0);
                qw[4 * v] = x.x;
                qw[4 * v + 1] = x.y;
                qw[4 * v + 2] = x.z;
                qw[4 * v + 3] = x.w;
            }
            auto qel = [&](int c) -> uint32_t {     // bf16 bits of channel 32tq + c
                return (qw[c >> 1] >> (16 * (c & 1))) & 0xffffu;
            };
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int b = 16 * (ks >> 2), i0 = 2 * (ks & 3);
                qf[ks][0] = bf16x2_to_f16x2(qel(b + i0), qel(b + i0 + 8));
                qf[ks][1] = bf16x2_to_f16x2(qel(b + i0 + 1), qel(b + i0 + 9));
            }
        }
        float o[8][4];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
            o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        float zp[4] = {0.f, 0.f, 0.f, 0.f};      // zero term of the values: [channel group gq][heads h0, h1]
        float m0 = -INFINITY, m1 = -INFINITY, r0 = -INFINITY, r1 = -INFINITY;
        // the weight sum of one block of one head per lane (see the reduction
        // below): lanes gq = 0, 2, 4, 6 of each column write the per-block
        // log2-sum-exp of block (gq & 4 ? 1 : 0) of head (gq & 2 ? h1 : h0)
        const bool wb = gq & 4, wh = gq & 2;
        float lpart = 0.f;
        float *lse_w = nullptr;
        if (!(gq & 1) && (wh ? h1 : h0) < G)
            lse_w = a.w.lse_blk + (static_cast<size_t>(it.l) * g.Hq + kvh * G + (wh ? h1 : h0)) * nb_total +
                    it.lse0 + (wb ? 1 : 0);

        for (uint32_t gi = 0; gi < it.ng; ++gi) {
            mbar_wait(smem_u32(&bars[warp][rg.st_cons]), rg.ph_cons, a.w.err);
            const uint32_t base = ring_u32 + rg.st_cons * kTile;
            // ---- S^T = K . Q^T for both blocks of the group (16 tokens x 8
            // heads each), two independent MMA chains.  A key is
            // fp16(code * s_c + z_c): the code, exact as code/2, times 2 s_c
            // plus z_c in one f16 fused multiply-add (one rounding)
            float sj[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            {
                const uint4 kw0 = lds128(base + lane * 16), kw1 = lds128(base + (32 + lane) * 16);
                const uint32_t kw[2][4] = {{kw0.x, kw0.y, kw0.z, kw0.w}, {kw1.x, kw1.y, kw1.z, kw1.w}};
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    // (scale, zero) pairs of the k-step's channels (c, c+8) and (c+1, c+9)
                    const uint4 m = lds128(base + 2048 + (ks * 4 + tq) * 16);
                    const uint32_t sa = m.x, sb = m.z;        // 2 s (the tile holds 2s)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint32_t wd = kw[j][ks >> 1];
                        uint32_t a0, a1, a2, a3;
                        e2m1x4((ks & 1) ? ((wd >> 2) & kCodeMask) : (wd & kCodeMask), a0, a1, a2, a3);
                        mma_f16(sj[j], hfma2u(a0, sa, m.y), hfma2u(a1, sa, m.y), hfma2u(a2, sb, m.w),
                                hfma2u(a3, sb, m.w), qf[ks][0], qf[ks][1]);
                    }
                }
            }
            // one online-softmax update for the 32 tokens; the per-block
            // log2-sum-exps are taken against the same running max.  The
            // lanes' maxima are merged only when one of them exceeds the
            // running max (otherwise the running max stands)
            // The maxima are compared in raw score units (r0, r1; m0, m1 are the
            // same maxima in log2 units, r * scale_log2): rounding is monotonic,
            // so this moves exactly when the log2-unit comparison would, and
            // a group that does not move the max needs no scaling of it.
            const float lm0 = fmaxf(fmaxf(sj[0][0], sj[0][2]), fmaxf(sj[1][0], sj[1][2]));
            const float lm1 = fmaxf(fmaxf(sj[0][1], sj[0][3]), fmaxf(sj[1][1], sj[1][3]));
            float sc0 = 1.f, sc1 = 1.f;     // rescale factors: 2^0 unless the running max moved
            bool moved = false;
            if (__any_sync(0xffffffffu, lm0 > r0 || lm1 > r1)) {
                float b0 = lm0, b1 = lm1;
#pragma unroll
                for (int x = 4; x < 32; x <<= 1) {
                    b0 = fmaxf(b0, __shfl_xor_sync(0xffffffffu, b0, x));
                    b1 = fmaxf(b1, __shfl_xor_sync(0xffffffffu, b1, x));
                }
                r0 = fmaxf(r0, b0);
                r1 = fmaxf(r1, b1);
                const float mn0 = r0 * scale_log2, mn1 = r1 * scale_log2;
                sc0 = fast_exp2(m0 - mn0);
                sc1 = fast_exp2(m1 - mn1);
                m0 = mn0;
                m1 = mn1;
                moved = true;
            }
            float pj[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                pj[j][0] = fast_exp2(fmaf(sj[j][0], scale_log2, -m0));
                pj[j][1] = fast_exp2(fmaf(sj[j][1], scale_log2, -m1));
                pj[j][2] = fast_exp2(fmaf(sj[j][2], scale_log2, -m0));
                pj[j][3] = fast_exp2(fmaf(sj[j][3], scale_log2, -m1));
            }
            uint32_t pb[2][2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                pb[j][0] = movmatrix_t(pack_f16(pj[j][0], pj[j][1]));
                pb[j][1] = movmatrix_t(pack_f16(pj[j][2], pj[j][3]));
            }
            // per-block sums of the (fp32) weights over the 8 lanes of a head's
            // column, reduced transposed: at each level a lane keeps half of
            // its sums and passes the other half, so that lane gq ends with
            // the sum of block (gq & 4) for head (gq & 2 ? h1 : h0)
            {
                const float w00 = pj[0][0] + pj[0][2], w01 = pj[0][1] + pj[0][3];   // block 0: h0, h1
                const float w10 = pj[1][0] + pj[1][2], w11 = pj[1][1] + pj[1][3];   // block 1
                float k0 = wb ? w10 : w00, k1 = wb ? w11 : w01;
                k0 += __shfl_xor_sync(0xffffffffu, wb ? w00 : w10, 16);
                k1 += __shfl_xor_sync(0xffffffffu, wb ? w01 : w11, 16);
                float v = wh ? k1 : k0;
                v += __shfl_xor_sync(0xffffffffu, wh ? k0 : k1, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                const float mnw = wh ? m1 : m0;
                lpart = lpart * (wh ? sc1 : sc0) + v;      // this lane's block of its head
                if (lse_w)
                    lse_w[2 * gi] = mnw + fast_log2(v);
            }
            // the rescale only after a merge of the maxima (otherwise every
            // factor is 2^0); `moved` is the same in every lane
            if (moved) {
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    o[mt][0] *= sc0;
                    o[mt][1] *= sc1;
                    o[mt][2] *= sc0;
                    o[mt][3] *= sc1;
                }
                zp[0] *= sc0;
                zp[1] *= sc1;
                zp[2] *= sc0;
                zp[3] *= sc1;
            }
            // ---- O^T += V^T . P^T per block.  Values are s_t * code + z_t per
            // token and 32-channel group: the codes (as code/2) against P^T
            // scaled by 2 s_t of the m-tile's channel group; the zero term,
            // one value per (channel group, head), by one MMA whose rows are
            // the four channel groups, into zp (added to O at the item's end)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint4 vw4 = lds128(base + 1024 + (j * 32 + lane) * 16);
                // 2 x scale pairs: token pairs tq and tq + 4, channel groups 0..3
                uint32_t vs[2][4];
#pragma unroll
                for (int hp = 0; hp < 2; ++hp) {
                    const uint4 x = lds128(base + 2560 + ((j * 8 + tq + 4 * hp) * 4) * 4);
                    vs[hp][0] = x.x; vs[hp][1] = x.y; vs[hp][2] = x.z; vs[hp][3] = x.w;
                }
                // zero pairs of channel group gq (A row gq; rows 4..15 zero):
                // token pairs tq and tq + 4
                const uint32_t za = base + 2816 + ((j * 8 + tq) * 4 + (gq & 3)) * 4;
                uint32_t z0 = lds32(za), z2 = lds32(za + 4 * 4 * 4);
                if (gq >= 4)
                    z0 = z2 = 0;
                if (j == 1) {
                    // every lane has read the tile: refill the stage
                    __syncwarp();
                    --rg.inflight;
                    if (++rg.st_cons == kKRing) {
                        rg.st_cons = 0;
                        rg.ph_cons ^= 1u;
                    }
                    if (rg.inflight < kKRing)
                        kissue_next(a, cur, nxt, have_nxt, c_in_nxt, c_grp, rg, ring_u32, bars[warp], lane);
                }
                const uint32_t vw[4] = {vw4.x, vw4.y, vw4.z, vw4.w};
#pragma unroll
                for (int cg = 0; cg < 4; ++cg) {
                    // P^T times 2 s_t (the tile holds 2s) of the channel group
                    const uint32_t b0 = hmul2u(pb[j][0], vs[0][cg]), b1 = hmul2u(pb[j][1], vs[1][cg]);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int mt = 2 * cg + half;
                        uint32_t a0, a1, a2, a3;
                        e2m1x4(half ? ((vw[cg] >> 2) & kCodeMask) : (vw[cg] & kCodeMask), a0, a1, a2, a3);
                        mma_f16(o[mt], a0, a1, a2, a3, b0, b1);
                    }
                }
                mma_f16(zp, z0, 0u, z2, 0u, pb[j][0], pb[j][1]);
            }
            if (gi == claim_at && !have_nxt) {
                nxt = prepare_kitem(a, claim(), lane);
                have_nxt = true;
                while (rg.inflight < kKRing &&
                       kissue_next(a, cur, nxt, have_nxt, c_in_nxt, c_grp, rg, ring_u32, bars[warp], lane)) {
                }
            }
        }

        // the values' zero term: channel group cg's (head h0, h1) sums sit in
        // lane 4 cg + tq; every channel of the group receives them
#pragma unroll
        for (int cg = 0; cg < 4; ++cg) {
            const float v0 = __shfl_sync(0xffffffffu, zp[0], 4 * cg + tq);
            const float v1 = __shfl_sync(0xffffffffu, zp[1], 4 * cg + tq);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                o[2 * cg + half][0] += v0;
                o[2 * cg + half][1] += v1;
                o[2 * cg + half][2] += v0;
                o[2 * cg + half][3] += v1;
            }
        }
        // the heads' weight sums: both blocks' parts (lanes 16 apart), then
        // head h1's from lane gq = 2 to lane gq = 0
        const float lhead = lpart + __shfl_xor_sync(0xffffffffu, lpart, 16);
        const float l1 = __shfl_xor_sync(0xffffffffu, lhead, 8), l0 = lhead;
        const uint32_t part = it.part;
        if (gq == 0) {
            a.w.part_ml[part * kMaxGroup + h0] = make_float2(m0, l0);
            a.w.part_ml[part * kMaxGroup + h1] = make_float2(m1, l1);
        }
        float *po = a.w.part_o + static_cast<size_t>(part) * kMaxGroup * kKD;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            po[h0 * kKD + mt * 16 + gq] = o[mt][0];
            po[h1 * kKD + mt * 16 + gq] = o[mt][1];
            po[h0 * kKD + mt * 16 + gq + 8] = o[mt][2];
            po[h1 * kKD + mt * 16 + gq + 8] = o[mt][3];
        }
        if (!have_nxt)                      // not claimed in the loop: claim now
            nxt = prepare_kitem(a, claim(), lane);
        if (c_in_nxt)
            c_in_nxt = false;
        else
            c_grp = 0;
        cur = nxt;
        have_nxt = false;
        nxt.it.valid = 0;
        nxt.it.ng = 0;
        while (cur.it.valid && rg.inflight < kKRing &&
               kissue_next(a, cur, nxt, have_nxt, c_in_nxt, c_grp, rg, ring_u32, bars[warp], lane)) {
        }
    }
}

constexpr size_t kKSmem = static_cast<size_t>(kKWarps) * kKRing * kTile + 128;

}  // namespace

cudaError_t launch_kivi_compress(const Geo &g, const KiviJob *jobs, uint32_t njobs, const uint8_t *pool,
                                 uint8_t *gpool, int32_t *table, cudaStream_t s)
{
    if (njobs == 0)
        return cudaSuccess;
    kivi_compress_kernel<<<njobs * g.L * g.Hkv, 128, 0, s>>>(g, jobs, pool, gpool, table);
    return cudaGetLastError();
}

int decode_kivi_blocks_per_sm(const Geo &)
{
    int n = 0;
    cudaFuncSetAttribute(decode_kivi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kKSmem));
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kivi_kernel, 32 * kKWarps, kKSmem);
    return n;
}

cudaError_t launch_decode_kivi(const Geo &g, const Work &w, const uint16_t *q, const int32_t *table,
                               const uint8_t *gpool, uint32_t n_items, int grid, cudaStream_t s)
{
    if (n_items == 0)
        return cudaSuccess;
    KArgs a{g, w, q, table, gpool, n_items};
    const int need = static_cast<int>((n_items + kKWarps - 1) / kKWarps);
    return launch_pdl(decode_kivi_kernel, dim3(need < grid ? need : grid), dim3(32 * kKWarps), kKSmem, s, a);
}

}  // namespace kvs
