// Host layer of the C ABI: configuration checks, free list and reference
// counts of the page pool, per-sequence block tables, the identity-keyed
// store of demoted blocks, the pinned upload ring and the launch sequence of
// every call.
//
// Sources: "LLM KV cache offload" (block manager, block tables, reference
// counts freeing a shared block only with its last user, demotion through
// pinned host staging on the copy engines); "GQA per-head attention as
// scoring streams" (identity key and score persist across eviction and are
// restored on re-admission); "RETRACTIONS" s.2 (blocks are write-once).
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <thread>

#include <nvtx3/nvToolsExt.h>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <map>
#include <memory>
#include <string>
#include <unordered_map>
#include <utility>
#include <vector>

#include <cudaTypedefs.h>

#include "kvs_internal.h"
#include "kvs_launch.h"

using namespace kvs;

// NVTX range around a public call (visible in Nsight Systems / Compute).
struct KvsRange {
    explicit KvsRange(const char *name) { nvtxRangePushA(name); }
    ~KvsRange() { nvtxRangePop(); }
};
#define KVS_RANGE() const KvsRange kvs_range_(__func__)

namespace {

constexpr uint32_t kRingSlots = 32;
constexpr size_t kRingSlotBytes = size_t(1) << 20;
constexpr size_t kReadbackBytes = 16384;            // header + first copy-list entries

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

uint64_t splitmix64(uint64_t &s)
{
    uint64_t z = (s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

struct SeqState {
    uint64_t id = 0;
    bool live = false;
    uint32_t ntok = 0;
    uint32_t shared_blocks = 0;      // leading blocks shared read-only
    uint32_t qtok = 0;               // KIVI: tokens held in 2-bit group pages
    std::vector<int32_t> table;      // page per block, -1 = demoted, KVS_TABLE_GROUP(g) = in group page g
};

struct Demoted {
    kvs_record rec;
    uint64_t host_off;
    uint32_t chunk;       // staging chunk whose device->host copy holds the page
};

}  // namespace

struct kvs_ctx {
    kvs_config cfg{};
    Geo geo{};
    Layout lay{};
    Work work{};
    kvs_buffers buf{};
    kvs_sizes sz{};
    int device = 0;
    int sm_count = 0;
    int decode_grid = 0;
    uint32_t wg = 1;
    alignas(64) CUtensorMap tmap;

    std::vector<SeqState> seqs;                     // by slot
    std::unordered_map<uint64_t, uint32_t> slot_of;
    std::vector<uint32_t> free_slots;
    std::deque<int32_t> free_pages;
    std::vector<uint32_t> refcnt;
    bool refcnt_dirty = true;                       // device mirror needs an upload
    std::map<std::pair<uint64_t, uint64_t>, Demoted> store;
    uint64_t t = 0;

    std::unique_ptr<DSet> dset;                     // host copy of the current set
    bool have_set = false;
    bool set_scored = false;     // the current set was scored by kvs_decode_score_step

    uint8_t *ring_host = nullptr;                   // pinned upload ring
    cudaEvent_t ring_ev[kRingSlots]{};
    bool ring_used[kRingSlots]{};
    uint32_t ring_next = 0;
    uint32_t *pinned_small = nullptr;               // readbacks
    uint32_t *async_hdr = nullptr;                  // counts of the latest ASYNC select, [4]: its tag
    uint32_t *async_hdr_dev = nullptr;              // ... its device mapping (kernels write it)
    cudaEvent_t ev_async{};                         // ... on the host after this event, or
    uint32_t async_seq = 0;                         // ... once async_hdr[4] holds this number
    bool async_tagged = false;                      //     (mirror selects: no event in the stream)
    cudaStream_t async_stream{};                    //     written by a kernel on this stream
    int async_kind = 0;                             // 0 none yet, 1 mirror, 2 ids only

    cudaEvent_t ev_ready[2]{}, ev_side_done{}, ev_pool_release{};
    cudaEvent_t ev_dec_start = nullptr, ev_dec_stop = nullptr;   // caller's timing events
    std::vector<cudaEvent_t> chunk_ev;              // end of each list-mode D2H chunk
    std::vector<int32_t> quarantine;                // demoted pages still being gathered
    cudaEvent_t ev_quarantine{};                    // after the gathers reading them
    bool side_pending = false, release_pending = false;

    uint64_t kernel_launches = 0;                   // kernels launched by this context
    std::deque<uint32_t> free_groups;               // KIVI: free group pages
    int kivi_grid = 0;                              // KIVI: persistent decode grid
    cudaEvent_t ev_wait{};                          // bounded host waits
    std::string err;

    // Releases what the context holds, also after a failed kvs_create.
    ~kvs_ctx()
    {
        for (auto &e : ring_ev)
            if (e)
                cudaEventDestroy(e);
        for (auto e : {ev_ready[0], ev_ready[1], ev_side_done, ev_pool_release, ev_quarantine, ev_wait, ev_async})
            if (e)
                cudaEventDestroy(e);
        for (auto e : chunk_ev)
            cudaEventDestroy(e);
        if (ring_host)
            cudaFreeHost(ring_host);
        if (pinned_small)
            cudaFreeHost(pinned_small);
        if (async_hdr)
            cudaFreeHost(async_hdr);
    }
};

namespace {

// Process-wide test hooks (kvs_debug_inject): a failing pinned allocation in
// the next kvs_create, and host waits that never see their event complete.
std::atomic<uint32_t> g_faults{0};
std::atomic<uint32_t> g_wait_limit_ms{600000};

// Text of the last failure of a call without a context (kvs_required_sizes,
// kvs_create) on this thread; kvs_last_error(NULL) returns it.
thread_local std::string t_err;

int fail(kvs_ctx *c, int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (c)
        c->err = buf;
    else
        t_err = buf;
    return code;
}

#define CU(call)                                                                         \
    do {                                                                                 \
        cudaError_t e_ = (call);                                                         \
        if (e_ != cudaSuccess)                                                           \
            return fail(ctx, KVS_ECUDA, "%s: %s (%s:%d)", #call, cudaGetErrorString(e_), \
                        __FILE__, __LINE__);                                             \
    } while (0)

// Waits on the host until `ev` has completed, polling with a limit:
// KVS_ETIMEOUT when the limit passes first (the device work stays enqueued),
// KVS_ECUDA for an error reported by the event.
int event_wait(kvs_ctx *ctx, cudaEvent_t ev, const char *what)
{
    const auto t0 = std::chrono::steady_clock::now();
    const auto limit = std::chrono::milliseconds(g_wait_limit_ms.load());
    for (uint32_t spin = 0;; ++spin) {
        cudaError_t e = (g_faults.load() & KVS_FAULT_WAIT) ? cudaErrorNotReady : cudaEventQuery(ev);
        if (e == cudaSuccess)
            return KVS_OK;
        if (e != cudaErrorNotReady)
            return fail(ctx, KVS_ECUDA, "%s: %s", what, cudaGetErrorString(e));
        if (std::chrono::steady_clock::now() - t0 > limit)
            return fail(ctx, KVS_ETIMEOUT, "%s: no completion within %u ms", what, g_wait_limit_ms.load());
        if (spin > 256)
            std::this_thread::yield();
    }
}

// Waits, as event_wait does, until a kernel enqueued on stream s has written
// `seq` into the pinned word *tag (acquire: what the kernel wrote before it is
// visible after).  The stream is queried now and then (a query is not a
// stream operation): an error on it ends the wait, and so does a stream that
// has drained without the tag.
int tag_wait(kvs_ctx *ctx, const uint32_t *tag, uint32_t seq, cudaStream_t s, const char *what)
{
    const auto t0 = std::chrono::steady_clock::now();
    const auto limit = std::chrono::milliseconds(g_wait_limit_ms.load());
    const bool faked = g_faults.load() & KVS_FAULT_WAIT;
    for (uint32_t spin = 0;; ++spin) {
        if (!faked && __atomic_load_n(tag, __ATOMIC_ACQUIRE) == seq)
            return KVS_OK;
        if (!faked && (spin & 255u) == 255u) {
            const cudaError_t e = cudaStreamQuery(s);
            if (e == cudaSuccess && __atomic_load_n(tag, __ATOMIC_ACQUIRE) != seq)
                return fail(ctx, KVS_EDEVICE, "%s: the stream drained without the completion word", what);
            if (e != cudaSuccess && e != cudaErrorNotReady)
                return fail(ctx, KVS_ECUDA, "%s: %s", what, cudaGetErrorString(e));
        }
        if (std::chrono::steady_clock::now() - t0 > limit)
            return fail(ctx, KVS_ETIMEOUT, "%s: no completion within %u ms", what, g_wait_limit_ms.load());
        if (spin > 256)
            std::this_thread::yield();
    }
}

// Waits for the work enqueued on `s` so far (event_wait on a fresh record).
int stream_wait(kvs_ctx *ctx, cudaStream_t s, const char *what)
{
    CU(cudaEventRecord(ctx->ev_wait, s));
    return event_wait(ctx, ctx->ev_wait, what);
}
#define WAIT(s)                                                  \
    do {                                                         \
        if (int rc_ = stream_wait(ctx, (s), __func__))           \
            return rc_;                                          \
    } while (0)

cudaStream_t S(void *s) { return static_cast<cudaStream_t>(s); }

struct RingSlot {
    uint32_t idx;
    uint8_t *host;
    uint8_t *dev;
};

// Takes the next ring slot (waiting for its previous user to finish).
int ring_acquire(kvs_ctx *ctx, size_t bytes, RingSlot *out)
{
    if (bytes > kRingSlotBytes)
        return fail(ctx, KVS_EINVAL, "upload of %zu bytes exceeds the ring slot (%zu)", bytes,
                    kRingSlotBytes);
    // the next slot whose last consumer is done; block only if all are busy
    uint32_t i = ctx->ring_next;
    for (uint32_t k = 0; k < kRingSlots; ++k) {
        const uint32_t j = (ctx->ring_next + k) % kRingSlots;
        if (!ctx->ring_used[j] || cudaEventQuery(ctx->ring_ev[j]) == cudaSuccess) {
            i = j;
            break;
        }
    }
    ctx->ring_next = (i + 1) % kRingSlots;
    if (ctx->ring_used[i])
        if (int rc = event_wait(ctx, ctx->ring_ev[i], "upload ring slot"))
            return rc;
    out->idx = i;
    out->host = ctx->ring_host + i * kRingSlotBytes;
    out->dev = ctx->work.ring + i * kRingSlotBytes;
    return KVS_OK;
}

// Copies the slot's bytes to its device side on `s` (after the host filled it).
int ring_push(kvs_ctx *ctx, const RingSlot &r, size_t bytes, cudaStream_t s)
{
    CU(cudaMemcpyAsync(r.dev, r.host, bytes, cudaMemcpyHostToDevice, s));
    return KVS_OK;
}

// Marks the slot busy until `s` passes this point (after its consumers).
int ring_release(kvs_ctx *ctx, const RingSlot &r, cudaStream_t s)
{
    CU(cudaEventRecord(ctx->ring_ev[r.idx], s));
    ctx->ring_used[r.idx] = true;
    return KVS_OK;
}

// Orders page writes on `s` after device->host copies still reading pages
// and after the release of pages by kvs_seq_remove.
int order_pool_writes(kvs_ctx *ctx, cudaStream_t s)
{
    if (ctx->side_pending)
        CU(cudaStreamWaitEvent(s, ctx->ev_side_done, 0));
    if (ctx->release_pending)
        CU(cudaStreamWaitEvent(s, ctx->ev_pool_release, 0));
    return KVS_OK;
}

// Makes `need` pages available on the free list for a writer on stream s.
// Pages demoted by a list-mode gather wait in quarantine until the gather
// kernels that read them have run: they return to the free list when that
// is known to be done, or, if the writer needs them now, after s is ordered
// behind those kernels.
int reclaim_pages(kvs_ctx *ctx, cudaStream_t s, size_t need)
{
    if (ctx->quarantine.empty())
        return KVS_OK;
    const bool done = cudaEventQuery(ctx->ev_quarantine) == cudaSuccess;
    if (!done && ctx->free_pages.size() >= need)
        return KVS_OK;
    if (!done)
        CU(cudaStreamWaitEvent(s, ctx->ev_quarantine, 0));
    for (int32_t p : ctx->quarantine)
        ctx->free_pages.push_back(p);
    ctx->quarantine.clear();
    return KVS_OK;
}

size_t pages_available(const kvs_ctx *ctx)
{
    return ctx->free_pages.size() + ctx->quarantine.size();
}

int check_cfg(const kvs_config *c, kvs_ctx *ctx)
{
    if (!c)
        return fail(ctx, KVS_EINVAL, "null config");
    if (c->block_tokens != KVS_BLOCK_TOKENS)
        return fail(ctx, KVS_EINVAL, "block_tokens must be 16");
    if (c->head_dim != 64 && c->head_dim != 128)
        return fail(ctx, KVS_EINVAL, "head_dim must be 64 or 128");
    if (!c->num_layers || !c->num_kv_heads || !c->num_q_heads ||
        c->num_q_heads % c->num_kv_heads)
        return fail(ctx, KVS_EINVAL, "head counts: Hq must be a positive multiple of Hkv");
    if (c->num_q_heads / c->num_kv_heads > static_cast<uint32_t>(kMaxGroup))
        return fail(ctx, KVS_EINVAL, "at most 8 query heads per KV head");
    if (!c->pool_blocks || !c->max_seqs || !c->max_blocks_per_seq || !c->staging_pages)
        return fail(ctx, KVS_EINVAL, "pool_blocks, max_seqs, max_blocks_per_seq, staging_pages must be > 0");
    if (static_cast<uint64_t>(c->num_layers) * c->pool_blocks >= (1ull << 31))
        return fail(ctx, KVS_EINVAL, "layers * pool_blocks must stay below 2^31");
    if (!(c->alpha >= 0.0 && c->alpha <= 1.0) || !c->recency_window)
        return fail(ctx, KVS_EINVAL, "alpha must be in [0, 1] and recency_window > 0");
    if (!(c->cut_lo <= c->cut_hi))
        return fail(ctx, KVS_EINVAL, "cut_lo must not exceed cut_hi");
    if (c->kv_dtype != KVS_KV_BF16 && c->kv_dtype != KVS_KV_FP8_E4M3 && c->kv_dtype != KVS_KV_KIVI2)
        return fail(ctx, KVS_EINVAL, "unknown kv_dtype %u", c->kv_dtype);
    if (c->kv_dtype == KVS_KV_KIVI2) {
        if (c->head_dim != 128)
            return fail(ctx, KVS_EINVAL, "2-bit groups need head_dim 128");
    }
    if (c->kv_dtype == KVS_KV_FP8_E4M3) {
        if (c->head_dim != 128)
            return fail(ctx, KVS_EINVAL, "FP8 pages need head_dim 128");
        if (!(c->k_scale > 0.f && c->k_scale < 1e30f && c->v_scale > 0.f && c->v_scale < 1e30f))
            return fail(ctx, KVS_EINVAL, "FP8 scales must be positive and finite");
    }
    return KVS_OK;
}

uint32_t pick_wg(uint32_t hkv)
{
    for (uint32_t w : {4u, 2u, 1u})
        if (hkv % w == 0)
            return w;
    return 1;
}

// KIVI: tokens in whole groups that end at least KVS_KIVI_RESIDUAL tokens
// before the end of an n-token sequence.
uint32_t kivi_q(uint64_t n)
{
    return n > KVS_KIVI_RESIDUAL
               ? static_cast<uint32_t>((n - KVS_KIVI_RESIDUAL) / KVS_KIVI_GROUP_TOKENS * KVS_KIVI_GROUP_TOKENS)
               : 0u;
}

SeqState *find_seq(kvs_ctx *ctx, uint64_t id, uint32_t *slot = nullptr)
{
    auto it = ctx->slot_of.find(id);
    if (it == ctx->slot_of.end())
        return nullptr;
    if (slot)
        *slot = it->second;
    return &ctx->seqs[it->second];
}

// Builds the decode set for seq_ids (call order); validates residency.
int build_set(kvs_ctx *ctx, const uint64_t *ids, uint32_t nseq, DSet *ds)
{
    if (!ids || nseq == 0 || nseq > kMaxCallSeqs)
        return fail(ctx, KVS_EINVAL, "nseq must be in [1, %u]", kMaxCallSeqs);
    std::memset(ds, 0, dset_bytes(nseq));
    const Geo &g = ctx->geo;
    uint32_t blk = 0, items = 0, items_q = 0, parts = 0;
    std::vector<std::pair<uint64_t, uint32_t>> order;
    order.reserve(nseq);
    uint32_t nres[kMaxCallSeqs], qbs[kMaxCallSeqs];
    for (uint32_t i = 0; i < nseq; ++i) {
        SeqState *s = find_seq(ctx, ids[i]);
        const uint32_t nb = s ? (s->ntok + kBlockTokens - 1) / kBlockTokens : 1;
        qbs[i] = s && g.kivi ? s->qtok / kBlockTokens : 0;
        nres[i] = nb - qbs[i];
    }
    // 2-bit group-page chunks (for the 2-bit decode kernel's warps), then the
    // page chunks with whatever partials are left
    PageChunks qc{kMinChunk, kMinChunk, 0};
    uint64_t parts_q = 0;
    if (g.kivi) {
        qc = pick_page_chunks(qbs, nseq, g.L, g.Hkv, static_cast<uint32_t>(ctx->kivi_grid) * 4,
                              ctx->lay.parts_max, 0);
        if (qc.big == 0)
            return fail(ctx, KVS_EINVAL, "too many blocks in one call for the workspace partials");
        for (uint32_t i = 0; i < nseq; ++i)
            parts_q += static_cast<uint64_t>(g.L) * g.Hkv * qc.nchunk(qbs[i]);
    }
    const PageChunks pc = pick_page_chunks(nres, nseq, g.L, g.Hkv, ctx->decode_grid * ctx->wg,
                                           ctx->lay.parts_max, parts_q);
    if (pc.big == 0)
        return fail(ctx, KVS_EINVAL, "too many blocks in one call for the workspace partials");
    for (uint32_t i = 0; i < nseq; ++i) {
        uint32_t slot;
        SeqState *s = find_seq(ctx, ids[i], &slot);
        if (!s)
            return fail(ctx, KVS_ENOTFOUND, "unknown sequence %llu", (unsigned long long)ids[i]);
        if (s->ntok == 0)
            return fail(ctx, KVS_EINVAL, "sequence %llu has no tokens", (unsigned long long)ids[i]);
        for (int32_t p : s->table)
            if (p == -1)
                return fail(ctx, KVS_EINVAL, "sequence %llu has a demoted block; re-admit it first",
                            (unsigned long long)ids[i]);
        DSeq &q = ds->seq[i];
        q.slot = slot;
        q.ntok = s->ntok;
        q.nb = (s->ntok + kBlockTokens - 1) / kBlockTokens;
        // KIVI: the leading qb blocks (group pages) and the rest (pages) are
        // chunked apart: group-page chunks first, then page chunks
        q.qb = g.kivi ? s->qtok / kBlockTokens : 0;
        q.nchunk_q = qc.nchunk(q.qb);
        q.nbig_q = qc.nbig(q.qb);
        const uint32_t nchunk_p = pc.nchunk(q.nb - q.qb);
        q.nbig = pc.nbig(q.nb - q.qb);
        q.nchunk = q.nchunk_q + nchunk_p;
        q.blk_off = blk;
        q.item_off = items;
        q.item_off_q = items_q;
        q.part_off = parts;
        q.seq_id = ids[i];
        blk += q.nb;
        items += g.L * g.Hkv * nchunk_p;      // one item per KV head and chunk
        items_q += g.L * g.Hkv * q.nchunk_q;
        parts += g.L * g.Hkv * q.nchunk;
        order.emplace_back(ids[i], i);
    }
    std::sort(order.begin(), order.end());
    for (uint32_t i = 1; i < nseq; ++i)
        if (order[i].first == order[i - 1].first)
            return fail(ctx, KVS_EINVAL, "sequence %llu listed twice",
                        (unsigned long long)order[i].first);
    if (blk > ctx->lay.nb_max)
        return fail(ctx, KVS_EINVAL, "%u blocks in one call exceed max_call_blocks %u", blk,
                    ctx->lay.nb_max);
    if (parts > ctx->lay.parts_max)
        return fail(ctx, KVS_EINVAL, "too many decode partials (%u > %u)", parts, ctx->lay.parts_max);
    uint32_t off = 0;
    for (uint32_t i = 0; i < nseq; ++i) {
        ds->seq[i].srt_ci = order[i].second;
        ds->seq[i].srt_off = off;
        off += ds->seq[order[i].second].nb;
    }
    ds->nseq = nseq;
    ds->nb_total = blk;
    ds->n_items = items;
    ds->n_items_q = items_q;
    ds->n_parts = parts;
    ds->wg = ctx->wg;
    ds->chunk = qc.big;
    ds->chunk_q_small = qc.small;
    ds->chunk_big = pc.big;
    ds->chunk_small = pc.small;
    ds->t = ctx->t;
    return KVS_OK;
}

int launch_rc(kvs_ctx *ctx, cudaError_t e, const char *what, uint32_t kernels = 1)
{
    if (e != cudaSuccess)
        return fail(ctx, KVS_ECUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
    ctx->kernel_launches += kernels;
    return KVS_OK;
}

// The header and the call's entries: a small set in a kernel's parameters,
// a larger one through the upload ring.
int upload_set(kvs_ctx *ctx, const DSet &ds, cudaStream_t s)
{
    const size_t bytes = dset_bytes(ds.nseq);
    if (bytes <= kSetInlineBytes)
        return launch_rc(ctx, launch_set(&ds, bytes, ctx->work.dset, s), "decode set");
    RingSlot r;
    int rc = ring_acquire(ctx, bytes, &r);
    if (rc)
        return rc;
    std::memcpy(r.host, &ds, bytes);
    CU(cudaMemcpyAsync(ctx->work.dset, r.host, bytes, cudaMemcpyHostToDevice, s));
    return ring_release(ctx, r, s);
}


// Patch list upload + kernel (table entries and records).
int apply_patches(kvs_ctx *ctx, const std::vector<Patch> &p, cudaStream_t s)
{
    const size_t per = kRingSlotBytes / sizeof(Patch);
    for (size_t a = 0; a < p.size(); a += per) {
        const size_t n = std::min(per, p.size() - a);
        RingSlot r;
        int rc = ring_acquire(ctx, n * sizeof(Patch), &r);
        if (rc)
            return rc;
        std::memcpy(r.host, p.data() + a, n * sizeof(Patch));
        if ((rc = ring_push(ctx, r, n * sizeof(Patch), s)))
            return rc;
        if ((rc = launch_rc(ctx,
                            launch_patch(ctx->geo, static_cast<int32_t *>(ctx->buf.block_table),
                                         static_cast<kvs_record *>(ctx->buf.records),
                                         ctx->work.page_clean, reinterpret_cast<const Patch *>(r.dev),
                                         static_cast<uint32_t>(n), s),
                            "patch")))
            return rc;
        if ((rc = ring_release(ctx, r, s)))
            return rc;
    }
    return KVS_OK;
}

// KIVI: quantises, on stream s, every group of the listed sequences (slot,
// state) that has fallen behind the residual window, then returns the
// groups' bf16 pages to the free list (later writers run after the kernel
// on the same stream).  The caller checked that enough group pages are free.
int kivi_compress(kvs_ctx *ctx, const std::vector<std::pair<uint32_t, SeqState *>> &seqs, cudaStream_t s)
{
    std::vector<KiviJob> jobs;
    for (const auto &e : seqs) {
        SeqState *sq = e.second;
        const uint32_t qn = kivi_q(sq->ntok);
        for (uint32_t t0 = sq->qtok; t0 < qn; t0 += KVS_KIVI_GROUP_TOKENS) {
            const uint32_t gi = t0 / KVS_KIVI_GROUP_TOKENS;
            KiviJob j{};
            j.slot = e.first;
            j.group = gi;
            j.page0 = sq->table[2 * gi];
            j.page1 = sq->table[2 * gi + 1];
            j.gpage = ctx->free_groups.front();
            ctx->free_groups.pop_front();
            jobs.push_back(j);
        }
    }
    if (jobs.empty())
        return KVS_OK;
    // on a failure the group pages go back; the bf16 pages stay in use
    auto undo = [&](int rc) {
        for (auto it = jobs.rbegin(); it != jobs.rend(); ++it)
            ctx->free_groups.push_front(it->gpage);
        return rc;
    };
    int rc = order_pool_writes(ctx, s);
    if (rc)
        return undo(rc);
    const uint32_t per_slot = static_cast<uint32_t>(kRingSlotBytes / sizeof(KiviJob));
    for (size_t off = 0; off < jobs.size(); off += per_slot) {
        const uint32_t n = static_cast<uint32_t>(std::min<size_t>(per_slot, jobs.size() - off));
        RingSlot r;
        if ((rc = ring_acquire(ctx, n * sizeof(KiviJob), &r)))
            return undo(rc);
        std::memcpy(r.host, jobs.data() + off, n * sizeof(KiviJob));
        if ((rc = ring_push(ctx, r, n * sizeof(KiviJob), s)))
            return undo(rc);
        if ((rc = launch_rc(ctx,
                            launch_kivi_compress(ctx->geo, reinterpret_cast<const KiviJob *>(r.dev), n,
                                                 static_cast<const uint8_t *>(ctx->buf.pool),
                                                 static_cast<uint8_t *>(ctx->buf.group_pool),
                                                 static_cast<int32_t *>(ctx->buf.block_table), s),
                            "2-bit compress")))
            return undo(rc);
        if ((rc = ring_release(ctx, r, s)))
            return undo(rc);
    }
    for (const KiviJob &j : jobs) {
        for (int32_t p : {j.page0, j.page1})
            if (--ctx->refcnt[p] == 0)
                ctx->free_pages.push_back(p);
    }
    size_t k = 0;
    for (const auto &e : seqs) {
        SeqState *sq = e.second;
        const uint32_t qn = kivi_q(sq->ntok);
        for (uint32_t t0 = sq->qtok; t0 < qn; t0 += KVS_KIVI_GROUP_TOKENS, ++k) {
            const uint32_t gi = t0 / KVS_KIVI_GROUP_TOKENS;
            sq->table[2 * gi] = KVS_TABLE_GROUP(jobs[k].gpage);
            sq->table[2 * gi + 1] = KVS_TABLE_GROUP(jobs[k].gpage);
        }
        sq->qtok = qn;
    }
    ctx->refcnt_dirty = true;
    return KVS_OK;
}

// KIVI: group pages a sequence of ntok_after tokens would take beyond what it holds.
uint32_t kivi_groups_needed(const SeqState *sq, uint64_t ntok_after)
{
    const uint32_t qn = kivi_q(ntok_after);
    return qn > sq->qtok ? (qn - sq->qtok) / KVS_KIVI_GROUP_TOKENS : 0u;
}

// The staging ring: with 4 pages or more, the gather double-buffers through
// its first two quarters and re-admission through the last two, so the two
// directions can run at once; below that the gather uses halves and
// re-admission copies page by page.
struct StagingSplit {
    uint32_t H;         // pages per buffer
    int nbuf;           // gather buffers (1 or 2)
    bool readmit_ring;  // re-admission has its own two buffers at 2H, 3H
};

StagingSplit staging_split(uint32_t C)
{
    if (C >= 4)
        return {C / 4, 2, true};
    if (C >= 2)
        return {C / 2, 2, false};
    return {1, 1, false};
}

kvs_record fresh_record(uint64_t seq_id, uint64_t b, uint64_t t)
{
    kvs_record r;
    std::memset(&r, 0, sizeof r);
    r.key.seq_id = seq_id;
    r.key.block_idx = b;
    r.last_touch = t;
    r.tier = 255;
    return r;
}

}  // namespace

// ---------------------------------------------------------------- layout

namespace kvs {

Layout workspace_layout(const kvs_config &c)
{
    Layout L{};
    const size_t nb_max = c.max_call_blocks ? c.max_call_blocks
                                            : static_cast<size_t>(c.max_seqs) * c.max_blocks_per_seq;
    const size_t seqs = std::min<size_t>(c.max_seqs, kMaxCallSeqs);
    const size_t LH = static_cast<size_t>(c.num_layers) * c.num_q_heads;
    L.nb_max = static_cast<uint32_t>(nb_max);
    // partials for chunks of 32 blocks, plus the short chunks at the end of
    // each stream: their blocks cover about one large chunk (at most 128
    // blocks) per decode warp (at most 2,048 warps), in chunks of 16, plus a
    // short remainder per stream
    L.parts_max = static_cast<uint32_t>(static_cast<size_t>(c.num_layers) * c.num_kv_heads *
                                            ((nb_max + 31) / 32 + 3 * seqs) +
                                        2048 * 128 / 16);
    L.tiles_max = static_cast<uint32_t>((nb_max + 1023) / 1024 + 1);
    L.ring_slots = kRingSlots;
    L.ring_slot_bytes = kRingSlotBytes;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.err = take(64);
    L.counter = take(64);
    L.sel_count = take(64);
    L.sel_thr = take(64);
    L.dset = take(sizeof(DSet));
    L.part_ml = take(static_cast<size_t>(L.parts_max) * kMaxGroup * sizeof(float2));
    L.part_o = take(static_cast<size_t>(L.parts_max) * kMaxGroup * c.head_dim * sizeof(float));
    L.lse_blk = take(LH * nb_max * sizeof(float));
    L.stream_mass = take(static_cast<size_t>(c.num_layers) * c.num_kv_heads * nb_max * sizeof(float));
    L.tile_cnt = take(L.tiles_max * sizeof(uint32_t));
    L.sel_ids = take(nb_max * sizeof(kvs_key));
    L.sel_pages = take(nb_max * sizeof(int32_t));
    L.sel_recidx = take(nb_max * sizeof(uint32_t));
    L.sel_recs = take(nb_max * sizeof(kvs_record));
    L.sel_full = take(nb_max);
    L.dev_refcnt = take(static_cast<size_t>(c.pool_blocks) * 4);
    L.page_cnt = take(static_cast<size_t>(c.pool_blocks) * 4);
    L.page_first = take(static_cast<size_t>(c.pool_blocks) * 4);
    L.page_pos = take(static_cast<size_t>(c.pool_blocks) * 4);
    L.page_clean = take(c.pool_blocks);
    L.plan_pages = take(nb_max * 4);
    L.plan_slot = take(nb_max * 4);
    L.readback = take((4 + nb_max) * 4);
    L.ring = take(kRingSlots * kRingSlotBytes);
    L.total = o;
    return L;
}

Work carve(const Layout &L, void *ws)
{
    uint8_t *b = static_cast<uint8_t *>(ws);
    Work w{};
    w.err = reinterpret_cast<uint32_t *>(b + L.err);
    w.err_info = w.err + 1;
    w.counter = reinterpret_cast<uint32_t *>(b + L.counter);
    w.sel_count = reinterpret_cast<uint32_t *>(b + L.sel_count);
    w.sel_thr = reinterpret_cast<uint64_t *>(b + L.sel_thr);
    w.dset = reinterpret_cast<DSet *>(b + L.dset);
    w.part_ml = reinterpret_cast<float2 *>(b + L.part_ml);
    w.part_o = reinterpret_cast<float *>(b + L.part_o);
    w.lse_blk = reinterpret_cast<float *>(b + L.lse_blk);
    w.stream_mass = reinterpret_cast<float *>(b + L.stream_mass);
    w.tile_cnt = reinterpret_cast<uint32_t *>(b + L.tile_cnt);
    w.sel_ids = reinterpret_cast<kvs_key *>(b + L.sel_ids);
    w.sel_pages = reinterpret_cast<int32_t *>(b + L.sel_pages);
    w.sel_recidx = reinterpret_cast<uint32_t *>(b + L.sel_recidx);
    w.sel_recs = reinterpret_cast<kvs_record *>(b + L.sel_recs);
    w.sel_full = b + L.sel_full;
    w.dev_refcnt = reinterpret_cast<uint32_t *>(b + L.dev_refcnt);
    w.page_cnt = reinterpret_cast<uint32_t *>(b + L.page_cnt);
    w.page_first = reinterpret_cast<uint32_t *>(b + L.page_first);
    w.page_pos = reinterpret_cast<int32_t *>(b + L.page_pos);
    w.page_clean = b + L.page_clean;
    w.plan_pages = reinterpret_cast<int32_t *>(b + L.plan_pages);
    w.plan_slot = reinterpret_cast<int32_t *>(b + L.plan_slot);
    w.readback = reinterpret_cast<uint32_t *>(b + L.readback);
    w.ring = b + L.ring;
    return w;
}

}  // namespace kvs

// ------------------------------------------------------------------ ABI

extern "C" {

int kvs_required_sizes(const kvs_config *cfg, kvs_sizes *out)
{
    KVS_RANGE();
    kvs_ctx *ctx = nullptr;
    int rc = check_cfg(cfg, ctx);
    if (rc)
        return rc;
    if (!out)
        return KVS_EINVAL;
    const kvs_config &c = *cfg;
    const size_t rows = static_cast<size_t>(c.max_seqs) * c.max_blocks_per_seq;
    const size_t elem = c.kv_dtype == KVS_KV_FP8_E4M3 ? 1 : 2;
    out->page_bytes = static_cast<size_t>(2) * c.num_layers * c.num_kv_heads * KVS_BLOCK_TOKENS *
                      c.head_dim * elem;
    out->pool_bytes = out->page_bytes * c.pool_blocks;
    out->table_bytes = rows * sizeof(int32_t);
    out->records_bytes = rows * sizeof(kvs_record);
    out->mass_bytes = rows * sizeof(float);
    out->workspace_bytes = workspace_layout(c).total;
    out->staging_bytes = out->page_bytes * c.staging_pages;
    const bool kivi = c.kv_dtype == KVS_KV_KIVI2;
    out->group_page_bytes = kivi ? static_cast<size_t>(c.num_layers) * c.num_kv_heads * KVS_KIVI_TILE_BYTES : 0;
    out->group_pool_bytes = out->group_page_bytes * (kivi ? c.kivi_groups : 0);
    return KVS_OK;
}

int kvs_create(const kvs_config *cfg, const kvs_buffers *buf, kvs_ctx_t **out)
{
    KVS_RANGE();
    if (!out)
        return KVS_EINVAL;
    *out = nullptr;
    std::unique_ptr<kvs_ctx> holder(new kvs_ctx());
    kvs_ctx *ctx = holder.get();
    struct KeepErr {            // a failed create leaves its text for kvs_last_error(NULL)
        std::unique_ptr<kvs_ctx> &h;
        ~KeepErr()
        {
            if (h)
                t_err = h->err;
        }
    } keep{holder};
    int rc = check_cfg(cfg, ctx);
    if (rc)
        return rc;
    if (!buf || !buf->pool || !buf->block_table || !buf->records || !buf->mass || !buf->workspace ||
        !buf->staging)
        return fail(ctx, KVS_EINVAL, "every device buffer must be given");
    for (void *p : {buf->pool, buf->block_table, buf->records, buf->mass, buf->workspace, buf->staging})
        if (reinterpret_cast<uintptr_t>(p) % 256)
            return fail(ctx, KVS_EINVAL, "device buffers must be 256-byte aligned");
    if (cfg->kv_dtype == KVS_KV_KIVI2 && cfg->kivi_groups &&
        (!buf->group_pool || reinterpret_cast<uintptr_t>(buf->group_pool) % 256))
        return fail(ctx, KVS_EINVAL, "2-bit groups need a 256-byte aligned group_pool");
    static_assert(sizeof(kvs_record) == KVS_RECORD_BYTES, "record must be 64 bytes");
    static_assert(sizeof(kvs_key) == 16, "key must be 16 bytes");
    ctx->cfg = *cfg;
    ctx->buf = *buf;
    kvs_required_sizes(cfg, &ctx->sz);
    ctx->lay = workspace_layout(*cfg);
    ctx->work = carve(ctx->lay, buf->workspace);
    Geo &g = ctx->geo;
    g.L = cfg->num_layers;
    g.Hq = cfg->num_q_heads;
    g.Hkv = cfg->num_kv_heads;
    g.d = cfg->head_dim;
    g.G = g.Hq / g.Hkv;
    g.pool_blocks = cfg->pool_blocks;
    g.max_seqs = cfg->max_seqs;
    g.mb = cfg->max_blocks_per_seq;
    g.page_bytes = ctx->sz.page_bytes;
    g.fp8 = cfg->kv_dtype == KVS_KV_FP8_E4M3 ? 1 : 0;
    g.k_scale = g.fp8 ? cfg->k_scale : 1.f;
    g.v_scale = g.fp8 ? cfg->v_scale : 1.f;
    g.kivi = cfg->kv_dtype == KVS_KV_KIVI2 ? 1 : 0;
    g.kivi_groups = g.kivi ? cfg->kivi_groups : 0;
    g.group_page_bytes = ctx->sz.group_page_bytes;
    for (uint32_t i = 0; i < g.kivi_groups; ++i)
        ctx->free_groups.push_back(i);
    ctx->wg = pick_wg(g.Hkv);
    ctx->dset.reset(new DSet());

    CU(cudaGetDevice(&ctx->device));
    CU(cudaDeviceGetAttribute(&ctx->sm_count, cudaDevAttrMultiProcessorCount, ctx->device));
    const int per_sm = decode_blocks_per_sm(g, ctx->wg);
    if (per_sm < 1)
        return fail(ctx, KVS_ECUDA, "decode kernel does not fit on an SM (%zu B shared memory)",
                    decode_smem_bytes(g, ctx->wg));
    ctx->decode_grid = per_sm * ctx->sm_count;
    if (g.kivi) {
        const int kper = decode_kivi_blocks_per_sm(g);
        if (kper < 1)
            return fail(ctx, KVS_ECUDA, "2-bit group decode kernel does not fit on an SM");
        ctx->kivi_grid = kper * ctx->sm_count;
    }

    // TMA descriptor of the pool: dims (d, token slot, KV head, K/V, layer*page)
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    cudaDriverEntryPointQueryResult qres;
    CU(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", reinterpret_cast<void **>(&encode),
                                        12000, cudaEnableDefault, &qres));
    if (qres != cudaDriverEntryPointSuccess || !encode)
        return fail(ctx, KVS_ECUDA, "cuTensorMapEncodeTiled not available");
    // bf16: 64-element (128-byte) boxes, two per row; FP8: one 128-byte box
    const cuuint64_t d = g.d, el = g.fp8 ? 1 : 2;
    cuuint64_t dims[5] = {d, KVS_BLOCK_TOKENS, g.Hkv, 2, static_cast<cuuint64_t>(g.L) * g.pool_blocks};
    cuuint64_t strides[4] = {d * el, KVS_BLOCK_TOKENS * d * el, g.Hkv * KVS_BLOCK_TOKENS * d * el,
                             2ull * g.Hkv * KVS_BLOCK_TOKENS * d * el};
    cuuint32_t box[5] = {g.fp8 ? 128u : 64u, KVS_BLOCK_TOKENS, 1, 2, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult cr = encode(&ctx->tmap, g.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         5, buf->pool, dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS)
        return fail(ctx, KVS_ECUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(cr));

    CU(cudaMemset(buf->block_table, 0xff, ctx->sz.table_bytes));
    CU(cudaMemset(buf->records, 0, ctx->sz.records_bytes));
    CU(cudaMemset(buf->mass, 0, ctx->sz.mass_bytes));
    CU(cudaMemset(buf->workspace, 0, ctx->lay.dset));   // error word, counters
    CU(cudaMemset(ctx->work.page_cnt, 0, static_cast<size_t>(cfg->pool_blocks) * 4));
    CU(cudaMemset(ctx->work.page_first, 0xff, static_cast<size_t>(cfg->pool_blocks) * 4));
    CU(cudaMemset(ctx->work.page_clean, 0, cfg->pool_blocks));
    CU(cudaMemset(ctx->work.dev_refcnt, 0, static_cast<size_t>(cfg->pool_blocks) * 4));
    if (g_faults.fetch_and(~KVS_FAULT_HOSTALLOC) & KVS_FAULT_HOSTALLOC)
        return fail(ctx, KVS_ENOMEM, "pinned host allocation failed (injected)");
    CU(cudaHostAlloc(reinterpret_cast<void **>(&ctx->ring_host), kRingSlots * kRingSlotBytes,
                     cudaHostAllocDefault));
    CU(cudaEventCreateWithFlags(&ctx->ev_wait, cudaEventDisableTiming));
    CU(cudaHostAlloc(reinterpret_cast<void **>(&ctx->pinned_small), kReadbackBytes, cudaHostAllocDefault));
    CU(cudaHostAlloc(reinterpret_cast<void **>(&ctx->async_hdr), 64, cudaHostAllocMapped));
    std::memset(ctx->async_hdr, 0, 64);
    CU(cudaHostGetDevicePointer(reinterpret_cast<void **>(&ctx->async_hdr_dev), ctx->async_hdr, 0));
    CU(cudaEventCreateWithFlags(&ctx->ev_async, cudaEventDisableTiming));
    for (auto &e : ctx->ring_ev)
        CU(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    for (int i = 0; i < 2; ++i) {
        CU(cudaEventCreateWithFlags(&ctx->ev_ready[i], cudaEventDisableTiming));
    }
    CU(cudaEventCreateWithFlags(&ctx->ev_side_done, cudaEventDisableTiming));
    CU(cudaEventCreateWithFlags(&ctx->ev_pool_release, cudaEventDisableTiming));
    CU(cudaEventCreateWithFlags(&ctx->ev_quarantine, cudaEventDisableTiming));
    CU(cudaDeviceSynchronize());

    ctx->seqs.resize(cfg->max_seqs);
    for (uint32_t i = cfg->max_seqs; i > 0; --i)
        ctx->free_slots.push_back(i - 1);
    std::vector<int32_t> perm(cfg->pool_blocks);
    for (uint32_t i = 0; i < cfg->pool_blocks; ++i)
        perm[i] = static_cast<int32_t>(i);
    uint64_t st = cfg->pool_seed;
    for (uint32_t i = cfg->pool_blocks; i > 1; --i) {   // Fisher-Yates
        const uint32_t j = static_cast<uint32_t>(splitmix64(st) % i);
        std::swap(perm[i - 1], perm[j]);
    }
    ctx->free_pages.assign(perm.begin(), perm.end());
    ctx->refcnt.assign(cfg->pool_blocks, 0);
    *out = holder.release();
    return KVS_OK;
}

void kvs_destroy(kvs_ctx_t *ctx)
{
    KVS_RANGE();
    if (!ctx)
        return;
    cudaDeviceSynchronize();
    delete ctx;
}

const char *kvs_last_error(const kvs_ctx_t *ctx) { return ctx ? ctx->err.c_str() : t_err.c_str(); }

int kvs_seq_add(kvs_ctx_t *ctx, uint64_t seq_id, int64_t parent, uint32_t shared_blocks, void *stream)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    if (ctx->slot_of.count(seq_id))
        return fail(ctx, KVS_EEXIST, "sequence %llu exists", (unsigned long long)seq_id);
    if (ctx->free_slots.empty())
        return fail(ctx, KVS_ENOMEM, "no free sequence slot (max_seqs %u)", ctx->cfg.max_seqs);
    SeqState *par = nullptr;
    if (shared_blocks && ctx->geo.kivi)
        return fail(ctx, KVS_EINVAL, "2-bit group contexts share no blocks");
    if (parent >= 0) {
        par = find_seq(ctx, static_cast<uint64_t>(parent));
        if (!par)
            return fail(ctx, KVS_ENOTFOUND, "parent %lld not found", (long long)parent);
        if (par->ntok / kBlockTokens < shared_blocks)
            return fail(ctx, KVS_EINVAL, "parent has %u full blocks, %u requested",
                        par->ntok / kBlockTokens, shared_blocks);
        for (uint32_t b = 0; b < shared_blocks; ++b)
            if (par->table[b] < 0)
                return fail(ctx, KVS_EINVAL, "parent block %u is demoted", b);
    } else if (shared_blocks) {
        return fail(ctx, KVS_EINVAL, "shared blocks need a parent");
    }
    if (shared_blocks > ctx->cfg.max_blocks_per_seq)
        return fail(ctx, KVS_EINVAL, "shared prefix longer than a table row");
    const uint32_t slot = ctx->free_slots.back();
    std::vector<Patch> patches;
    for (uint32_t b = 0; b < shared_blocks; ++b) {
        Patch p{};
        p.slot = slot;
        p.block = b;
        p.page = par->table[b];
        p.what = kPatchRecord;
        p.rec = fresh_record(seq_id, b, ctx->t);
        patches.push_back(p);
    }
    if (!patches.empty()) {
        int rc = apply_patches(ctx, patches, S(stream));
        if (rc)
            return rc;
    }
    ctx->free_slots.pop_back();
    SeqState &s = ctx->seqs[slot];
    s = SeqState();
    s.id = seq_id;
    s.live = true;
    s.shared_blocks = shared_blocks;
    for (uint32_t b = 0; b < shared_blocks; ++b) {
        s.table.push_back(par->table[b]);
        ctx->refcnt[par->table[b]] += 1;
    }
    ctx->refcnt_dirty = true;
    s.ntok = shared_blocks * kBlockTokens;
    ctx->slot_of[seq_id] = slot;
    return KVS_OK;
}

int kvs_seq_remove(kvs_ctx_t *ctx, uint64_t seq_id, void *stream)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    uint32_t slot;
    SeqState *s = find_seq(ctx, seq_id, &slot);
    if (!s)
        return fail(ctx, KVS_ENOTFOUND, "unknown sequence %llu", (unsigned long long)seq_id);
    CU(cudaEventRecord(ctx->ev_pool_release, S(stream)));
    ctx->release_pending = true;
    for (size_t b = 0; b < s->table.size(); ++b) {
        const int32_t p = s->table[b];
        if (p <= KVS_TABLE_GROUP(0)) {
            if (b % 2 == 0)                     // both blocks name the group page
                ctx->free_groups.push_back(static_cast<uint32_t>(KVS_TABLE_GROUP(0) - p));
            continue;
        }
        if (p < 0)
            continue;
        if (--ctx->refcnt[p] == 0)
            ctx->free_pages.push_back(p);
    }
    ctx->refcnt_dirty = true;
    for (auto it = ctx->store.begin(); it != ctx->store.end();)
        it = it->first.first == seq_id ? ctx->store.erase(it) : std::next(it);
    *s = SeqState();
    ctx->slot_of.erase(seq_id);
    ctx->free_slots.push_back(slot);
    if (ctx->have_set)
        for (uint32_t i = 0; i < ctx->dset->nseq; ++i)
            if (ctx->dset->seq[i].seq_id == seq_id)
                ctx->have_set = false;
    return KVS_OK;
}

int kvs_append_tokens(kvs_ctx_t *ctx, uint64_t seq_id, uint32_t n, const void *k_dev,
                      const void *v_dev, void *stream)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    uint32_t slot;
    SeqState *s = find_seq(ctx, seq_id, &slot);
    if (!s)
        return fail(ctx, KVS_ENOTFOUND, "unknown sequence %llu", (unsigned long long)seq_id);
    if (n == 0 || !k_dev || !v_dev)
        return fail(ctx, KVS_EINVAL, "append needs n > 0 and K/V pointers");
    if ((reinterpret_cast<uintptr_t>(k_dev) | reinterpret_cast<uintptr_t>(v_dev)) % 16)
        return fail(ctx, KVS_EINVAL, "K/V must be 16-byte aligned");
    const uint64_t p0 = s->ntok, p1 = p0 + n;
    const uint32_t first_blk = static_cast<uint32_t>(p0 / kBlockTokens);
    const uint64_t last_blk = (p1 - 1) / kBlockTokens;
    if (last_blk >= ctx->cfg.max_blocks_per_seq)
        return fail(ctx, KVS_EINVAL, "sequence would need %llu blocks (table row holds %u)",
                    (unsigned long long)(last_blk + 1), ctx->cfg.max_blocks_per_seq);
    const uint32_t nb_old = static_cast<uint32_t>((p0 + kBlockTokens - 1) / kBlockTokens);
    const uint32_t nblk = static_cast<uint32_t>(last_blk) - first_blk + 1;
    if (first_blk < nb_old) {
        if (first_blk < s->shared_blocks)
            return fail(ctx, KVS_EINVAL, "block %u is shared read-only", first_blk);
        if (s->table[first_blk] < 0)
            return fail(ctx, KVS_EINVAL, "block %u is demoted", first_blk);
    }
    const uint32_t need = static_cast<uint32_t>(last_blk + 1) - nb_old;
    if (pages_available(ctx) < need)
        return fail(ctx, KVS_ENOMEM, "pool exhausted: %u pages needed, %zu free", need,
                    pages_available(ctx));
    if (ctx->geo.kivi && kivi_groups_needed(s, p1) > ctx->free_groups.size())
        return fail(ctx, KVS_ENOMEM, "group pool exhausted: %u group pages needed, %zu free",
                    kivi_groups_needed(s, p1), ctx->free_groups.size());
    int rc = order_pool_writes(ctx, S(stream));
    if (rc || (rc = reclaim_pages(ctx, S(stream), need)))
        return rc;
    RingSlot r;
    if ((rc = ring_acquire(ctx, nblk * sizeof(int32_t), &r)))
        return rc;
    int32_t *pages = reinterpret_cast<int32_t *>(r.host);
    std::vector<int32_t> fresh;
    for (uint32_t b = first_blk; b <= last_blk; ++b) {
        if (b < nb_old) {
            pages[b - first_blk] = s->table[b];
        } else {
            pages[b - first_blk] = ctx->free_pages.front();
            fresh.push_back(ctx->free_pages.front());
            ctx->free_pages.pop_front();
        }
    }
    auto undo = [&]() {
        for (auto it = fresh.rbegin(); it != fresh.rend(); ++it)
            ctx->free_pages.push_front(*it);
    };
    if ((rc = ring_push(ctx, r, nblk * sizeof(int32_t), S(stream)))) {
        undo();
        return rc;
    }
    AppendArgs a{};
    a.k = static_cast<const uint16_t *>(k_dev);
    a.v = static_cast<const uint16_t *>(v_dev);
    a.pool = static_cast<uint16_t *>(ctx->buf.pool);
    a.page_clean = ctx->work.page_clean;
    a.table = static_cast<int32_t *>(ctx->buf.block_table);
    a.records = static_cast<kvs_record *>(ctx->buf.records);
    a.pages = reinterpret_cast<const int32_t *>(r.dev);
    a.slot = slot;
    a.p0 = static_cast<uint32_t>(p0);
    a.n = n;
    a.first_blk = first_blk;
    a.nblk = nblk;
    a.first_new = nb_old;
    a.seq_id = seq_id;
    a.t_create = ctx->t;
    if ((rc = launch_rc(ctx, launch_append(ctx->geo, a, S(stream)), "append"))) {
        undo();
        return rc;
    }
    if ((rc = ring_release(ctx, r, S(stream))))
        return rc;
    for (uint32_t b = first_blk; b <= last_blk; ++b) {
        const int32_t p = pages[b - first_blk];
        if (b >= nb_old) {
            s->table.push_back(p);
            ctx->refcnt[p] = 1;
            ctx->refcnt_dirty = true;
        }
    }
    s->ntok = static_cast<uint32_t>(p1);
    if (ctx->geo.kivi)
        return kivi_compress(ctx, {{slot, s}}, S(stream));
    return KVS_OK;
}

int kvs_append_token(kvs_ctx_t *ctx, uint64_t seq_id, const void *k_dev, const void *v_dev,
                     void *stream)
{
    KVS_RANGE();
    return kvs_append_tokens(ctx, seq_id, 1, k_dev, v_dev, stream);
}

int kvs_append_step(kvs_ctx_t *ctx, const uint64_t *seq_ids, uint32_t nseq, const void *k_dev,
                    const void *v_dev, void *stream)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    if (!seq_ids || nseq == 0 || nseq > kMaxCallSeqs || !k_dev || !v_dev)
        return fail(ctx, KVS_EINVAL, "append_step needs 1..%u sequences and K/V pointers", kMaxCallSeqs);
    if ((reinterpret_cast<uintptr_t>(k_dev) | reinterpret_cast<uintptr_t>(v_dev)) % 16)
        return fail(ctx, KVS_EINVAL, "K/V must be 16-byte aligned");
    const Geo &g = ctx->geo;
    std::vector<StepAppend> sa(nseq);
    std::vector<SeqState *> seqs(nseq);
    uint32_t fresh = 0;
    {
        std::vector<uint64_t> sorted(seq_ids, seq_ids + nseq);
        std::sort(sorted.begin(), sorted.end());
        for (uint32_t i = 1; i < nseq; ++i)
            if (sorted[i] == sorted[i - 1])
                return fail(ctx, KVS_EINVAL, "sequence %llu listed twice", (unsigned long long)sorted[i]);
    }
    for (uint32_t i = 0; i < nseq; ++i) {
        uint32_t slot;
        SeqState *s = find_seq(ctx, seq_ids[i], &slot);
        if (!s)
            return fail(ctx, KVS_ENOTFOUND, "unknown sequence %llu", (unsigned long long)seq_ids[i]);
        const uint32_t pos = s->ntok, b = pos / kBlockTokens;
        if (b >= ctx->cfg.max_blocks_per_seq)
            return fail(ctx, KVS_EINVAL, "sequence %llu: table row full", (unsigned long long)seq_ids[i]);
        if (pos % kBlockTokens) {
            if (b < s->shared_blocks)
                return fail(ctx, KVS_EINVAL, "block %u of %llu is shared read-only", b,
                            (unsigned long long)seq_ids[i]);
            if (s->table[b] < 0)
                return fail(ctx, KVS_EINVAL, "block %u of %llu is demoted", b, (unsigned long long)seq_ids[i]);
        } else {
            ++fresh;
        }
        seqs[i] = s;
        sa[i].slot = slot;
        sa[i].pos = pos;
        sa[i].seq_id = seq_ids[i];
    }
    if (pages_available(ctx) < fresh)
        return fail(ctx, KVS_ENOMEM, "pool exhausted: %u pages needed, %zu free", fresh, pages_available(ctx));
    if (ctx->geo.kivi) {
        size_t groups = 0;
        for (uint32_t i = 0; i < nseq; ++i)
            groups += kivi_groups_needed(seqs[i], seqs[i]->ntok + 1ull);
        if (groups > ctx->free_groups.size())
            return fail(ctx, KVS_ENOMEM, "group pool exhausted: %zu group pages needed, %zu free", groups,
                        ctx->free_groups.size());
    }
    int rc = order_pool_writes(ctx, S(stream));
    if (rc || (rc = reclaim_pages(ctx, S(stream), fresh)))
        return rc;
    uint32_t rows = 0;
    const uint32_t rows_per_slot = g.L * 2 * g.Hkv;
    std::vector<int32_t> taken;
    for (uint32_t i = 0; i < nseq; ++i) {
        const uint32_t pos = sa[i].pos;
        sa[i].fresh = pos % kBlockTokens == 0;
        if (sa[i].fresh) {
            sa[i].page = ctx->free_pages.front();
            ctx->free_pages.pop_front();
            taken.push_back(sa[i].page);
            sa[i].nslots = kBlockTokens;
        } else {
            sa[i].page = seqs[i]->table[pos / kBlockTokens];
            sa[i].nslots = 1;
        }
        sa[i].row_off = rows;
        rows += sa[i].nslots * rows_per_slot;
    }
    auto undo = [&]() {
        for (auto it = taken.rbegin(); it != taken.rend(); ++it)
            ctx->free_pages.push_front(*it);
    };
    // a few sequences: the entries go in the kernel's parameters; more go
    // through the upload ring
    const bool inline_args = nseq <= kStepInline;
    RingSlot r{};
    if (!inline_args) {
        if ((rc = ring_acquire(ctx, nseq * sizeof(StepAppend), &r))) {
            undo();
            return rc;
        }
        std::memcpy(r.host, sa.data(), nseq * sizeof(StepAppend));
        if ((rc = ring_push(ctx, r, nseq * sizeof(StepAppend), S(stream)))) {
            undo();
            return rc;
        }
    }
    if ((rc = launch_rc(ctx,
                        launch_append_step(g, static_cast<const uint16_t *>(k_dev),
                                           static_cast<const uint16_t *>(v_dev),
                                           static_cast<uint16_t *>(ctx->buf.pool),
                                           static_cast<int32_t *>(ctx->buf.block_table),
                                           static_cast<kvs_record *>(ctx->buf.records), ctx->work.page_clean,
                                           inline_args ? nullptr : reinterpret_cast<const StepAppend *>(r.dev),
                                           sa.data(), nseq, rows, ctx->t, S(stream)),
                        "append_step"))) {
        undo();
        return rc;
    }
    if (!inline_args && (rc = ring_release(ctx, r, S(stream))))
        return rc;
    for (uint32_t i = 0; i < nseq; ++i) {
        if (sa[i].fresh) {
            seqs[i]->table.push_back(sa[i].page);
            ctx->refcnt[sa[i].page] = 1;
            ctx->refcnt_dirty = true;
        }
        seqs[i]->ntok += 1;
    }
    if (ctx->geo.kivi) {
        std::vector<std::pair<uint32_t, SeqState *>> due;
        for (uint32_t i = 0; i < nseq; ++i)
            if (kivi_groups_needed(seqs[i], seqs[i]->ntok))
                due.emplace_back(sa[i].slot, seqs[i]);
        return kivi_compress(ctx, due, S(stream));
    }
    return KVS_OK;
}

}  // extern "C"

namespace {

ScoreArgs score_args(const kvs_ctx *ctx)
{
    const kvs_config &c = ctx->cfg;
    return ScoreArgs{c.alpha, c.w_recency, c.w_ema, c.w_anchor, c.cut_lo, c.cut_hi, c.recency_window};
}

// decode + combine + masses; with score, the epilogue also scores the set
int decode_impl(kvs_ctx_t *ctx, const uint64_t *seq_ids, uint32_t nseq, const void *q_dev, float *out_dev,
                void *stream, bool score)
{
    if (!q_dev || !out_dev)
        return fail(ctx, KVS_EINVAL, "q and out must be given");
    if ((reinterpret_cast<uintptr_t>(q_dev) | reinterpret_cast<uintptr_t>(out_dev)) % 16)
        return fail(ctx, KVS_EINVAL, "q and out must be 16-byte aligned");
    DSet *ds = ctx->dset.get();
    int rc = build_set(ctx, seq_ids, nseq, ds);
    if (rc) {
        ctx->have_set = false;
        return rc;
    }
    ctx->t += 1;
    ds->t = ctx->t;
    cudaStream_t s = S(stream);
    if ((rc = upload_set(ctx, *ds, s)))
        return rc;
    ctx->have_set = true;
    const int grid = static_cast<int>(std::min<uint32_t>((ds->n_items + ctx->wg - 1) / ctx->wg,
                                                         ctx->decode_grid));
    if (ctx->ev_dec_start)
        CU(cudaEventRecord(ctx->ev_dec_start, s));
    if (ds->n_items_q &&
        (rc = launch_rc(ctx,
                        launch_decode_kivi(ctx->geo, ctx->work, static_cast<const uint16_t *>(q_dev),
                                           static_cast<const int32_t *>(ctx->buf.block_table),
                                           static_cast<const uint8_t *>(ctx->buf.group_pool), ds->n_items_q,
                                           ctx->kivi_grid, s),
                        "2-bit decode")))
        return rc;
    if (ds->n_items &&
        (rc = launch_rc(ctx,
                        launch_decode(ctx->geo, ctx->tmap, ctx->work, static_cast<const uint16_t *>(q_dev),
                                      static_cast<const int32_t *>(ctx->buf.block_table), ds->n_items,
                                      ctx->wg, grid, s),
                        "decode")))
        return rc;
    if (ctx->ev_dec_stop)
        CU(cudaEventRecord(ctx->ev_dec_stop, s));
    uint32_t max_nb = 0, max_nchunk = 0;
    for (uint32_t i = 0; i < ds->nseq; ++i) {
        max_nb = std::max(max_nb, ds->seq[i].nb);
        max_nchunk = std::max(max_nchunk, ds->seq[i].nchunk);
    }
    if ((rc = launch_rc(ctx, launch_combine(ctx->geo, ctx->work, out_dev, ds->nseq, max_nb, max_nchunk,
                                            static_cast<uint32_t>(ctx->sm_count), s),
                        "combine")))
        return rc;
    const ScoreArgs sa = score_args(ctx);
    if ((rc = launch_rc(ctx,
                        launch_mass(ctx->geo, ctx->work, static_cast<float *>(ctx->buf.mass), ds->nb_total,
                                    static_cast<kvs_record *>(ctx->buf.records), score ? &sa : nullptr, s),
                        "mass")))
        return rc;
    ctx->set_scored = score;
    return KVS_OK;
}

}  // namespace

extern "C" {

int kvs_decode_step(kvs_ctx_t *ctx, const uint64_t *seq_ids, uint32_t nseq, const void *q_dev,
                    float *out_dev, void *stream)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    return decode_impl(ctx, seq_ids, nseq, q_dev, out_dev, stream, false);
}

int kvs_decode_score_step(kvs_ctx_t *ctx, const uint64_t *seq_ids, uint32_t nseq, const void *q_dev,
                          float *out_dev, void *stream)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    return decode_impl(ctx, seq_ids, nseq, q_dev, out_dev, stream, true);
}

int kvs_score_update(kvs_ctx_t *ctx, void *stream)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    if (!ctx->have_set)
        return fail(ctx, KVS_EINVAL, "no decode set: call kvs_decode_step first");
    if (ctx->set_scored)
        return fail(ctx, KVS_EINVAL, "the last decode set was scored by kvs_decode_score_step");
    const kvs_config &c = ctx->cfg;
    return launch_rc(ctx,
                     launch_score(ctx->geo, ctx->work, static_cast<kvs_record *>(ctx->buf.records),
                                  static_cast<const float *>(ctx->buf.mass), c.alpha, c.recency_window,
                                  c.w_recency, c.w_ema, c.w_anchor, c.cut_lo, c.cut_hi,
                                  ctx->dset->nb_total, S(stream)),
                     "score");
}

int kvs_set_alpha(kvs_ctx_t *ctx, double alpha)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    if (!(alpha >= 0.0 && alpha <= 1.0))
        return fail(ctx, KVS_EINVAL, "alpha must be in [0, 1]");
    ctx->cfg.alpha = alpha;
    return KVS_OK;
}

int kvs_select_and_gather(kvs_ctx_t *ctx, const kvs_gather_args *args, kvs_gather_result *res)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    if (!args || !res)
        return fail(ctx, KVS_EINVAL, "args and result must be given");
    std::memset(res, 0, sizeof *res);
    if (!ctx->have_set)
        return fail(ctx, KVS_EINVAL, "no decode set: call kvs_decode_step first");
    const bool mirror = args->flags & KVS_GATHER_MIRROR, demote = args->flags & KVS_GATHER_DEMOTE;
    const bool async = args->flags & KVS_GATHER_ASYNC;
    if (args->flags & ~(KVS_GATHER_MIRROR | KVS_GATHER_DEMOTE | KVS_GATHER_ASYNC))
        return fail(ctx, KVS_EINVAL, "unknown flags 0x%x", args->flags);
    if (mirror && demote)
        return fail(ctx, KVS_EINVAL, "DEMOTE works in list mode only");
    if (ctx->geo.kivi && ((args->flags & ~KVS_GATHER_ASYNC) || args->host_dst))
        return fail(ctx, KVS_EINVAL,
                    "2-bit group contexts return the selection only (no host_dst, flags 0 or ASYNC)");
    if (async && !mirror && !ctx->geo.kivi)
        return fail(ctx, KVS_EINVAL, "ASYNC works with MIRROR (or in a 2-bit context) only");
    if (args->mode != KVS_SELECT_THRESH && args->mode != KVS_SELECT_LOWFRAC && args->mode != KVS_SELECT_LRFU)
        return fail(ctx, KVS_EINVAL, "unknown selection mode %d", args->mode);
    const size_t pb = ctx->sz.page_bytes;
    if (mirror && (!args->host_dst || args->host_dst_bytes < pb * ctx->cfg.pool_blocks))
        return fail(ctx, KVS_EINVAL, "MIRROR needs host_dst of pool_blocks pages");
    if (args->mode != KVS_SELECT_THRESH && !(args->frac >= 0.0 && args->frac <= 1.0))
        return fail(ctx, KVS_EINVAL, "frac must be in [0, 1]");
    if (args->mode == KVS_SELECT_LRFU && !(ctx->cfg.alpha < 1.0))
        return fail(ctx, KVS_EINVAL, "LRFU needs alpha < 1 (the key slope -ln(1-alpha) is infinite)");
    // ASYNC mirror: the device address of host_dst (page-locked and mapped)
    void *host_dev = nullptr;
    if (async && mirror) {
        cudaPointerAttributes pa{};
        if (cudaPointerGetAttributes(&pa, args->host_dst) != cudaSuccess || pa.type != cudaMemoryTypeHost ||
            !pa.devicePointer) {
            cudaGetLastError();
            return fail(ctx, KVS_EINVAL, "ASYNC needs host_dst in page-locked memory the device can address");
        }
        host_dev = pa.devicePointer;
    }
    cudaStream_t s = S(args->stream);
    cudaStream_t side = args->side_stream ? S(args->side_stream) : s;
    const uint32_t N = ctx->dset->nb_total;
    const Work &w = ctx->work;
    int rc;

    // ---- device: reference counts, selection, gather plan ---------------
    if (ctx->refcnt_dirty) {
        RingSlot r;
        const size_t bytes = ctx->refcnt.size() * sizeof(uint32_t);
        if ((rc = ring_acquire(ctx, bytes, &r)))
            return rc;
        std::memcpy(r.host, ctx->refcnt.data(), bytes);
        CU(cudaMemcpyAsync(w.dev_refcnt, r.host, bytes, cudaMemcpyHostToDevice, s));
        if ((rc = ring_release(ctx, r, s)))
            return rc;
        ctx->refcnt_dirty = false;
    }
    bool run = true;
    const double alpha = ctx->cfg.alpha;     // LRFU: the kernels take the key's slope from it
    if (args->mode != KVS_SELECT_THRESH) {
        const uint32_t k = static_cast<uint32_t>(std::floor(args->frac * static_cast<double>(N)));
        if (k == 0)
            run = false;
        else if ((rc = launch_rc(ctx,
                                 launch_radix_select(ctx->geo, w, static_cast<const kvs_record *>(ctx->buf.records),
                                                     N, k, args->mode, alpha, s),
                                 "radix select")))
            return rc;
    }
    uint32_t nsel = 0, npages = 0, ncopy = 0;
    std::vector<uint32_t> copy_list;
    if (run) {
        // asynchronous calls: the kernels write the caller's lists and the
        // counts (through the pinned header's device mapping) themselves, so
        // no copy follows them
        const uint32_t cap = std::min(N, args->ids_capacity);
        SelectOut sel_out{};
        if (async && args->ids_dev) {
            sel_out.ids = args->ids_dev;
            sel_out.ids_cap = cap;
        }
        if (async && ctx->geo.kivi)
            sel_out.count_host = ctx->async_hdr_dev;
        const bool one_kernel = !ctx->geo.kivi && select_plan_fits(N);
        if (one_kernel) {
            // selection and plan in one launch
            SelectOut o = sel_out;
            if (async) {
                if (args->slot_dev) {
                    o.slots = args->slot_dev;
                    o.ids_cap = cap;
                }
                o.count_host = ctx->async_hdr_dev;
            }
            if ((rc = launch_rc(ctx,
                                launch_select_plan(ctx->geo, w, static_cast<const kvs_record *>(ctx->buf.records),
                                                   static_cast<const int32_t *>(ctx->buf.block_table), args->mode,
                                                   alpha, N, mirror ? 1u : 0u, o, s),
                                "select and plan")))
                return rc;
        } else if ((rc = launch_rc(ctx,
                                   launch_select(ctx->geo, w, static_cast<const kvs_record *>(ctx->buf.records),
                                                 static_cast<const int32_t *>(ctx->buf.block_table), args->mode,
                                                 alpha, N, !ctx->geo.kivi, sel_out, s),
                                   "select", select_launches(N))))
            return rc;
        if (ctx->geo.kivi && async) {
            CU(cudaEventRecord(ctx->ev_async, s));
            ctx->async_tagged = false;
            ctx->async_kind = 2;
            return KVS_OK;
        }
        if (ctx->geo.kivi) {
            // the id list only: quantised blocks have no page to plan
            CU(cudaMemcpyAsync(ctx->pinned_small, w.sel_count, 4, cudaMemcpyDeviceToHost, s));
            WAIT(s);
            nsel = ctx->pinned_small[0];
            res->n_selected = nsel;
            if (nsel && args->ids_dev)
                CU(cudaMemcpyAsync(args->ids_dev, w.sel_ids, std::min(nsel, args->ids_capacity) * sizeof(kvs_key),
                                   cudaMemcpyDeviceToDevice, s));
            return KVS_OK;
        }
        SelectOut plan_out{};
        if (async) {
            if (args->slot_dev) {
                plan_out.slots = args->slot_dev;
                plan_out.ids_cap = cap;
            }
            plan_out.count_host = ctx->async_hdr_dev;
        }
        if (!one_kernel && (rc = launch_rc(ctx, launch_plan(w, mirror ? 1u : 0u, plan_out, s), "plan")))
            return rc;
        if (async) {
            // the stale pages go to the host mirror by a device kernel in
            // stream order (writers after it need no wait); the plan kernel
            // wrote the counts into pinned memory, read by kvs_gather_counts
            // ... and, once those copies are visible here, the counts and
            // the call's number into async_hdr: no event in the stream, so
            // the next step's first kernel still launches programmatically
            const uint32_t seq = ctx->async_seq + 1;
            if ((rc = launch_rc(ctx,
                                launch_mirror_copy(ctx->geo, w, static_cast<const uint16_t *>(ctx->buf.pool),
                                                   host_dev, ctx->cfg.pool_blocks, 2 * ctx->sm_count,
                                                   ctx->async_hdr_dev, seq, s),
                                "mirror copy")))
                return rc;
            ctx->async_seq = seq;
            ctx->async_tagged = true;
            ctx->async_stream = s;
            ctx->async_kind = 1;
            return KVS_OK;
        }
        // one readback: counts and the head of the copy list
        CU(cudaMemcpyAsync(ctx->pinned_small, w.readback, kReadbackBytes, cudaMemcpyDeviceToHost, s));
        WAIT(s);
        nsel = ctx->pinned_small[0];
        npages = ctx->pinned_small[1];
        ncopy = ctx->pinned_small[2];
        const uint32_t head = static_cast<uint32_t>(kReadbackBytes / 4 - 4);
        copy_list.assign(ctx->pinned_small + 4, ctx->pinned_small + 4 + std::min(ncopy, head));
        if (ncopy > head) {
            copy_list.resize(ncopy);
            CU(cudaMemcpyAsync(copy_list.data() + head, w.readback + 4 + head, (ncopy - head) * 4,
                               cudaMemcpyDeviceToHost, s));
            WAIT(s);
        }
    }
    if (async) {
        // nothing to select (k = 0): zero counts, in stream order
        CU(cudaMemsetAsync(w.readback, 0, 16, s));
        CU(cudaMemcpyAsync(ctx->async_hdr, w.readback, 16, cudaMemcpyDeviceToHost, s));
        CU(cudaEventRecord(ctx->ev_async, s));
        ctx->async_tagged = false;
        ctx->async_kind = ctx->geo.kivi ? 2 : 1;
        return KVS_OK;
    }
    res->n_selected = nsel;
    res->n_pages = npages;
    if (nsel && args->ids_dev)
        CU(cudaMemcpyAsync(args->ids_dev, w.sel_ids, std::min(nsel, args->ids_capacity) * sizeof(kvs_key),
                           cudaMemcpyDeviceToDevice, s));
    if (nsel && args->slot_dev && !demote && !(!mirror && npages > (args->host_dst ? args->host_dst_bytes / pb : 0)))
        CU(cudaMemcpyAsync(args->slot_dev, w.plan_slot, std::min(nsel, args->ids_capacity) * sizeof(int32_t),
                           cudaMemcpyDeviceToDevice, s));

    uint8_t *host = static_cast<uint8_t *>(args->host_dst);
    uint32_t nstage = npages;
    bool trunc = false;
    if (mirror) {
        // ---- mirror: copy the stale pages straight from the pool ----------
        if (ncopy) {
            CU(cudaEventRecord(ctx->ev_ready[0], s));
            CU(cudaStreamWaitEvent(side, ctx->ev_ready[0], 0));
            const uint8_t *pool = static_cast<const uint8_t *>(ctx->buf.pool);
            for (uint32_t p : copy_list)
                CU(cudaMemcpyAsync(host + static_cast<size_t>(p) * pb, pool + static_cast<size_t>(p) * pb, pb,
                                   cudaMemcpyDeviceToHost, side));
            CU(cudaEventRecord(ctx->ev_side_done, side));
            ctx->side_pending = true;
        }
        res->n_staged = ncopy;
        res->bytes_to_host = static_cast<uint64_t>(ncopy) * pb;
        return KVS_OK;
    }

    // ---- list mode: plan pages through the staging ring, in order --------
    const size_t cap = args->host_dst ? args->host_dst_bytes / pb : 0;
    if (nstage > cap) {
        nstage = static_cast<uint32_t>(cap);
        trunc = true;
    }
    std::vector<int32_t> slots;
    std::vector<kvs_key> dids;
    std::vector<int32_t> dpages;
    std::vector<kvs_record> drecs;
    if ((trunc || demote) && nsel) {
        // small lists, read back before any copy is enqueued so this call
        // never waits for the device->host copies
        slots.resize(nsel);
        CU(cudaMemcpyAsync(slots.data(), w.plan_slot, nsel * sizeof(int32_t), cudaMemcpyDeviceToHost, s));
        if (demote && nstage) {
            dids.resize(nsel);
            dpages.resize(nsel);
            drecs.resize(nsel);
            CU(cudaMemcpyAsync(dids.data(), w.sel_ids, nsel * sizeof(kvs_key), cudaMemcpyDeviceToHost, s));
            CU(cudaMemcpyAsync(dpages.data(), w.sel_pages, nsel * sizeof(int32_t), cudaMemcpyDeviceToHost, s));
            CU(cudaMemcpyAsync(drecs.data(), w.sel_recs, nsel * sizeof(kvs_record), cudaMemcpyDeviceToHost, s));
        }
        WAIT(s);
        if (trunc)
            for (auto &x : slots)
                if (x >= static_cast<int32_t>(nstage))
                    x = -1;
        if (args->slot_dev) {
            const uint32_t n = std::min(nsel, args->ids_capacity);
            RingSlot r;
            if ((rc = ring_acquire(ctx, n * sizeof(int32_t), &r)))
                return rc;
            std::memcpy(r.host, slots.data(), n * sizeof(int32_t));
            CU(cudaMemcpyAsync(args->slot_dev, r.host, n * sizeof(int32_t), cudaMemcpyHostToDevice, s));
            if ((rc = ring_release(ctx, r, s)))
                return rc;
        }
    }
    const StagingSplit split = staging_split(ctx->cfg.staging_pages);
    if (nstage) {
        // the whole gather chain runs on the side stream: gather kernel into
        // a staging buffer, then its device->host copy; the main stream stays
        // free (re-admission can overlap the copies)
        const uint32_t H = split.H;
        const int nbuf = split.nbuf;
        uint8_t *staging = static_cast<uint8_t *>(ctx->buf.staging);
        CU(cudaEventRecord(ctx->ev_ready[0], s));        // selection and plan done
        CU(cudaStreamWaitEvent(side, ctx->ev_ready[0], 0));
        CU(cudaStreamWaitEvent(side, ctx->ev_side_done, 0));   // staging free of the last call
        for (uint32_t c0 = 0, ci = 0; c0 < nstage; c0 += H, ++ci) {
            const uint32_t cnt = std::min(H, nstage - c0);
            uint8_t *dst = staging + static_cast<size_t>(ci % nbuf) * H * pb;
            if ((rc = launch_rc(ctx,
                                launch_gather(ctx->geo, static_cast<const uint16_t *>(ctx->buf.pool),
                                              w.plan_pages + c0, cnt, dst, side),
                                "gather")))
                return rc;
            CU(cudaMemcpyAsync(host + static_cast<size_t>(c0) * pb, dst, static_cast<size_t>(cnt) * pb,
                               cudaMemcpyDeviceToHost, side));
            while (ctx->chunk_ev.size() <= ci) {
                cudaEvent_t e;
                CU(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
                ctx->chunk_ev.push_back(e);
            }
            CU(cudaEventRecord(ctx->chunk_ev[ci], side));
        }
        CU(cudaEventRecord(ctx->ev_side_done, side));
        if (!demote)
            ctx->side_pending = true;    // gathered pages stay live: writers wait
        res->n_staged = nstage;
        res->bytes_to_host = static_cast<uint64_t>(nstage) * pb;
    }

    // ---- demotion: keep records by key, clear table entries, free pages ---
    if (demote && nstage) {
        const std::vector<kvs_key> &ids = dids;
        const std::vector<int32_t> &pages = dpages;
        const std::vector<kvs_record> &recs = drecs;
        for (uint32_t i = 0; i < nsel; ++i) {
            if (slots[i] < 0)
                continue;
            const std::pair<uint64_t, uint64_t> key(ids[i].seq_id, ids[i].block_idx);
            if (ctx->store.count(key))
                return fail(ctx, KVS_EEXIST, "key (%llu, %llu) already demoted",
                            (unsigned long long)key.first, (unsigned long long)key.second);
        }
        std::vector<Patch> patches;
        for (uint32_t i = 0; i < nsel; ++i) {
            if (slots[i] < 0)
                continue;
            const std::pair<uint64_t, uint64_t> key(ids[i].seq_id, ids[i].block_idx);
            ctx->store[key] = Demoted{recs[i], static_cast<uint64_t>(slots[i]) * pb,
                                      static_cast<uint32_t>(slots[i]) / split.H};
            uint32_t slot;
            SeqState *sq = find_seq(ctx, ids[i].seq_id, &slot);
            const int32_t p = pages[i];
            sq->table[ids[i].block_idx] = -1;
            Patch q{};
            q.slot = slot;
            q.block = static_cast<uint32_t>(ids[i].block_idx);
            q.page = -1;
            q.what = kPatchRecord;
            q.rec = recs[i];
            q.rec.flags |= 1;
            patches.push_back(q);
            if (--ctx->refcnt[p] == 0)
                ctx->quarantine.push_back(p);   // free once the gathers have read it
            res->n_demoted += 1;
        }
        ctx->refcnt_dirty = true;
        CU(cudaEventRecord(ctx->ev_quarantine, side));
        if ((rc = apply_patches(ctx, patches, s)))
            return rc;
        ctx->have_set = false;   // the set now has holes
    }
    if (trunc)
        return fail(ctx, KVS_ETRUNC, "host_dst holds %u of %u pages", nstage, npages);
    return KVS_OK;
}

int kvs_gather_counts(kvs_ctx_t *ctx, kvs_gather_result *res)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    if (!res)
        return fail(ctx, KVS_EINVAL, "res must be given");
    std::memset(res, 0, sizeof *res);
    if (!ctx->async_kind)
        return fail(ctx, KVS_EINVAL, "no asynchronous select on this context");
    if (int rc = ctx->async_tagged ? tag_wait(ctx, ctx->async_hdr + 4, ctx->async_seq, ctx->async_stream,
                                              "kvs_gather_counts")
                                   : event_wait(ctx, ctx->ev_async, "kvs_gather_counts"))
        return rc;
    res->n_selected = ctx->async_hdr[0];
    if (ctx->async_kind == 1) {
        res->n_pages = ctx->async_hdr[1];
        res->n_staged = ctx->async_hdr[2];
        res->bytes_to_host = static_cast<uint64_t>(res->n_staged) * ctx->sz.page_bytes;
    }
    return KVS_OK;
}

}  // extern "C"

namespace {

// Re-admission of the demoted keys ks: validation, pages from the free list,
// host-to-device copies (in host order, or in the order of ks), records and
// table entries restored.  Nothing changes on an error.
int readmit_keys(kvs_ctx_t *ctx, std::vector<std::pair<uint64_t, uint64_t>> ks, bool host_order,
                 const void *host_src, size_t host_src_bytes, cudaStream_t s)
{
    const uint32_t n = static_cast<uint32_t>(ks.size());
    const size_t pb = ctx->sz.page_bytes;
    {
        auto sorted = ks;
        std::sort(sorted.begin(), sorted.end());
        for (uint32_t i = 1; i < n; ++i)
            if (sorted[i] == sorted[i - 1])
                return fail(ctx, KVS_EEXIST, "key (%llu, %llu) listed twice",
                            (unsigned long long)sorted[i].first, (unsigned long long)sorted[i].second);
    }
    for (auto &k : ks) {
        auto it = ctx->store.find(k);
        if (it == ctx->store.end()) {
            SeqState *sq = find_seq(ctx, k.first);
            if (sq && k.second < sq->table.size() && sq->table[k.second] >= 0)
                return fail(ctx, KVS_EEXIST, "key (%llu, %llu) is resident",
                            (unsigned long long)k.first, (unsigned long long)k.second);
            return fail(ctx, KVS_ENOTFOUND, "key (%llu, %llu) is not demoted",
                        (unsigned long long)k.first, (unsigned long long)k.second);
        }
        if (it->second.host_off + pb > host_src_bytes)
            return fail(ctx, KVS_EINVAL, "host_src too small for key (%llu, %llu)",
                        (unsigned long long)k.first, (unsigned long long)k.second);
    }
    if (pages_available(ctx) < n)
        return fail(ctx, KVS_ENOMEM, "pool exhausted: %u pages needed, %zu free", n,
                    pages_available(ctx));
    int rc = order_pool_writes(ctx, s);
    if (rc || (rc = reclaim_pages(ctx, s, n)))
        return rc;
    // copy in host order (or the given order) and wait only for the D2H
    // chunks that hold each page, so re-admission overlaps the tail of a
    // demotion still in flight
    if (host_order)
        std::sort(ks.begin(), ks.end(), [&](const std::pair<uint64_t, uint64_t> &x,
                                            const std::pair<uint64_t, uint64_t> &y) {
            return ctx->store.at(x).host_off < ctx->store.at(y).host_off;
        });
    std::vector<Patch> patches;
    std::vector<int32_t> taken;
    const uint8_t *src = static_cast<const uint8_t *>(host_src);
    for (auto &k : ks) {
        const Demoted &dm = ctx->store.at(k);
        taken.push_back(ctx->free_pages.front());
        ctx->free_pages.pop_front();
        uint32_t slot;
        find_seq(ctx, k.first, &slot);
        Patch q{};
        q.slot = slot;
        q.block = static_cast<uint32_t>(k.second);
        q.page = taken.back();
        q.what = kPatchRecord | kPatchPageWritten;
        q.rec = dm.rec;
        patches.push_back(q);
    }
    auto undo = [&]() {
        for (auto it = taken.rbegin(); it != taken.rend(); ++it)
            ctx->free_pages.push_front(*it);
    };
    const StagingSplit split = staging_split(ctx->cfg.staging_pages);
    int64_t waited = -1;
    auto wait_chunks = [&](uint32_t c0, uint32_t c1) -> int {
        for (uint32_t c = c0; c <= c1; ++c)
            if (static_cast<int64_t>(c) > waited && c < ctx->chunk_ev.size()) {
                CU(cudaStreamWaitEvent(s, ctx->chunk_ev[c], 0));
                waited = c;
            }
        return static_cast<int>(KVS_OK);
    };
    if (split.readmit_ring) {
        // runs of host-contiguous pages: one copy into the staging half, then
        // a kernel places each page into its new pool page
        const uint32_t R = 2 * split.H;
        uint8_t *buf = static_cast<uint8_t *>(ctx->buf.staging) + static_cast<size_t>(2 * split.H) * pb;
        RingSlot r;
        if ((rc = ring_acquire(ctx, taken.size() * sizeof(int32_t), &r))) {
            undo();
            return rc;
        }
        std::memcpy(r.host, taken.data(), taken.size() * sizeof(int32_t));
        if ((rc = ring_push(ctx, r, taken.size() * sizeof(int32_t), s))) {
            undo();
            return rc;
        }
        for (size_t i = 0; i < ks.size();) {
            const uint64_t off0 = ctx->store.at(ks[i]).host_off;
            size_t j = i + 1;
            while (j < ks.size() && j - i < R && ctx->store.at(ks[j]).host_off == off0 + (j - i) * pb)
                ++j;
            const uint32_t n = static_cast<uint32_t>(j - i);
            if (n == 1) {       // a lone page goes straight into its pool page
                if ((rc = wait_chunks(ctx->store.at(ks[i]).chunk, ctx->store.at(ks[i]).chunk))) {
                    undo();
                    return rc;
                }
                const cudaError_t e = cudaMemcpyAsync(
                    static_cast<uint8_t *>(ctx->buf.pool) + static_cast<size_t>(taken[i]) * pb, src + off0, pb,
                    cudaMemcpyHostToDevice, s);
                if (e != cudaSuccess) {
                    undo();
                    return fail(ctx, KVS_ECUDA, "readmit copy: %s", cudaGetErrorString(e));
                }
                i = j;
                continue;
            }
            if ((rc = wait_chunks(ctx->store.at(ks[i]).chunk, ctx->store.at(ks[j - 1]).chunk)) ||
                (rc = [&]() -> int {
                    CU(cudaMemcpyAsync(buf, src + off0, static_cast<size_t>(n) * pb, cudaMemcpyHostToDevice, s));
                    return static_cast<int>(KVS_OK);
                }()) ||
                (rc = launch_rc(ctx,
                                launch_scatter(ctx->geo, buf, reinterpret_cast<const int32_t *>(r.dev) + i, n,
                                               static_cast<uint16_t *>(ctx->buf.pool), s),
                                "scatter"))) {
                undo();
                return rc;
            }
            i = j;
        }
        if ((rc = ring_release(ctx, r, s)))
            return rc;
    } else {
        for (size_t i = 0; i < ks.size(); ++i) {
            const Demoted &dm = ctx->store.at(ks[i]);
            if ((rc = wait_chunks(dm.chunk, dm.chunk))) {
                undo();
                return rc;
            }
            cudaError_t e = cudaMemcpyAsync(static_cast<uint8_t *>(ctx->buf.pool) + static_cast<size_t>(taken[i]) * pb,
                                            src + dm.host_off, pb, cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess) {
                undo();
                return fail(ctx, KVS_ECUDA, "readmit copy: %s", cudaGetErrorString(e));
            }
        }
    }
    if ((rc = apply_patches(ctx, patches, s)))
        return rc;
    for (size_t i = 0; i < ks.size(); ++i) {
        uint32_t slot;
        SeqState *sq = find_seq(ctx, ks[i].first, &slot);
        sq->table[ks[i].second] = taken[i];
        ctx->refcnt[taken[i]] = 1;
        ctx->store.erase(ks[i]);
    }
    ctx->refcnt_dirty = true;
    return KVS_OK;
}

// Plan of kvs_prefetch_plan: the first min(budget, demoted) keys in fetch
// order and their order keys (class << 62 | (bits(1.0) - bits(blend))).
int prefetch_plan(kvs_ctx_t *ctx, uint32_t budget, std::vector<std::pair<uint64_t, uint64_t>> &plan,
                  std::vector<uint64_t> &pkeys, cudaStream_t s)
{
    plan.clear();
    pkeys.clear();
    std::vector<std::pair<uint64_t, uint64_t>> keys;
    std::vector<PrefCand> cands;
    for (const auto &e : ctx->store) {          // (seq_id, block_idx) order
        const SeqState *sq = find_seq(ctx, e.first.first);
        if (!sq)
            continue;
        cands.push_back(PrefCand{e.second.rec.score, sq->ntok, static_cast<uint32_t>(e.first.second)});
        keys.push_back(e.first);
    }
    const uint32_t n = static_cast<uint32_t>(cands.size());
    const uint32_t k = std::min(budget, n);
    if (k == 0)
        return KVS_OK;
    if (n > ctx->lay.nb_max)
        return fail(ctx, KVS_EINVAL, "%u demoted blocks exceed the plan workspace (%u)", n, ctx->lay.nb_max);
    // candidates in ring-slot pieces straight into the selection scratch,
    // idle outside kvs_select_and_gather
    PrefCand *dcand = reinterpret_cast<PrefCand *>(ctx->work.sel_recs);
    const uint32_t per_slot = static_cast<uint32_t>(kRingSlotBytes / sizeof(PrefCand));
    for (uint32_t off = 0; off < n; off += per_slot) {
        const uint32_t m = std::min(per_slot, n - off);
        RingSlot r;
        int rc = ring_acquire(ctx, m * sizeof(PrefCand), &r);
        if (rc)
            return rc;
        std::memcpy(r.host, cands.data() + off, m * sizeof(PrefCand));
        CU(cudaMemcpyAsync(dcand + off, r.host, m * sizeof(PrefCand), cudaMemcpyHostToDevice, s));
        if ((rc = ring_release(ctx, r, s)))
            return rc;
    }
    uint64_t *dkeys = reinterpret_cast<uint64_t *>(ctx->work.sel_ids);
    uint64_t *dout_key = dkeys + ctx->lay.nb_max;
    uint32_t *dout_idx = ctx->work.sel_recidx;
    int rc = launch_rc(ctx, launch_prefetch_plan(dcand, n, k, dkeys, dout_key, dout_idx, s), "prefetch plan");
    if (rc)
        return rc;
    std::vector<uint32_t> idx(k);
    pkeys.resize(k);
    CU(cudaMemcpyAsync(pkeys.data(), dout_key, k * sizeof(uint64_t), cudaMemcpyDeviceToHost, s));
    CU(cudaMemcpyAsync(idx.data(), dout_idx, k * sizeof(uint32_t), cudaMemcpyDeviceToHost, s));
    WAIT(s);
    plan.resize(k);
    for (uint32_t i = 0; i < k; ++i) {
        if (idx[i] >= n)
            return fail(ctx, KVS_ECUDA, "prefetch plan returned index %u of %u", idx[i], n);
        plan[i] = keys[idx[i]];
    }
    return KVS_OK;
}

int write_plan(const std::vector<std::pair<uint64_t, uint64_t>> &plan, const std::vector<uint64_t> &pkeys,
               kvs_key *keys_out, double *blend_out, uint8_t *class_out, uint32_t *n_out)
{
    for (size_t i = 0; i < plan.size(); ++i) {
        keys_out[i].seq_id = plan[i].first;
        keys_out[i].block_idx = plan[i].second;
        const uint64_t low = pkeys[i] & ((uint64_t(1) << 62) - 1);
        if (blend_out) {
            const uint64_t bits = 0x3FF0000000000000ull - low;
            std::memcpy(&blend_out[i], &bits, sizeof bits);
        }
        if (class_out)
            class_out[i] = static_cast<uint8_t>(pkeys[i] >> 62);
    }
    *n_out = static_cast<uint32_t>(plan.size());
    return KVS_OK;
}

}  // namespace

extern "C" {

int kvs_readmit(kvs_ctx_t *ctx, const kvs_key *keys, uint32_t n, const void *host_src,
                size_t host_src_bytes, void *stream)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    if (n == 0)
        return KVS_OK;
    if (!keys || !host_src)
        return fail(ctx, KVS_EINVAL, "keys and host_src must be given");
    std::vector<std::pair<uint64_t, uint64_t>> ks(n);
    for (uint32_t i = 0; i < n; ++i)
        ks[i] = {keys[i].seq_id, keys[i].block_idx};
    return readmit_keys(ctx, std::move(ks), true, host_src, host_src_bytes, S(stream));
}

int kvs_prefetch_plan(kvs_ctx_t *ctx, uint32_t budget, kvs_key *keys_out, double *blend_out,
                      uint8_t *class_out, uint32_t *n_out, void *stream)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    if (!keys_out || !n_out)
        return fail(ctx, KVS_EINVAL, "keys_out and n_out must be given");
    if (budget > KVS_PREFETCH_MAX)
        return fail(ctx, KVS_EINVAL, "budget %u exceeds %u", budget, KVS_PREFETCH_MAX);
    *n_out = 0;
    std::vector<std::pair<uint64_t, uint64_t>> plan;
    std::vector<uint64_t> pkeys;
    int rc = prefetch_plan(ctx, budget, plan, pkeys, S(stream));
    if (rc)
        return rc;
    return write_plan(plan, pkeys, keys_out, blend_out, class_out, n_out);
}

int kvs_prefetch(kvs_ctx_t *ctx, uint32_t budget, const void *host_src, size_t host_src_bytes,
                 kvs_key *keys_out, double *blend_out, uint8_t *class_out, uint32_t *n_out, void *stream)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    if (!keys_out || !n_out || !host_src)
        return fail(ctx, KVS_EINVAL, "keys_out, n_out and host_src must be given");
    if (budget > KVS_PREFETCH_MAX)
        return fail(ctx, KVS_EINVAL, "budget %u exceeds %u", budget, KVS_PREFETCH_MAX);
    *n_out = 0;
    cudaStream_t s = S(stream);
    std::vector<std::pair<uint64_t, uint64_t>> plan;
    std::vector<uint64_t> pkeys;
    int rc = prefetch_plan(ctx, budget, plan, pkeys, s);
    if (rc || plan.empty())
        return rc;
    if ((rc = readmit_keys(ctx, plan, false, host_src, host_src_bytes, s)))
        return rc;
    return write_plan(plan, pkeys, keys_out, blend_out, class_out, n_out);
}

int kvs_debug_set_mass(kvs_ctx_t *ctx, const uint64_t *seq_ids, uint32_t nseq, const float *mass_dev,
                       void *stream)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    if (!mass_dev)
        return fail(ctx, KVS_EINVAL, "mass must be given");
    DSet *ds = ctx->dset.get();
    int rc = build_set(ctx, seq_ids, nseq, ds);
    if (rc) {
        ctx->have_set = false;
        return rc;
    }
    ds->t = ctx->t;
    cudaStream_t s = S(stream);
    if ((rc = upload_set(ctx, *ds, s)))
        return rc;
    ctx->have_set = true;
    ctx->set_scored = false;
    return launch_rc(ctx,
                     launch_copy_mass(ctx->geo, ctx->work, mass_dev, static_cast<float *>(ctx->buf.mass),
                                      nseq, s),
                     "copy mass");
}

int kvs_debug_chunk_plan(const uint32_t *nres, uint32_t n, uint32_t num_layers, uint32_t num_kv_heads,
                         uint32_t workers, uint64_t parts_cap, uint64_t extra_parts, uint32_t *big,
                         uint32_t *small, uint32_t *tail)
{
    if (!nres || !big || !small || !tail || n == 0 || !num_layers || !num_kv_heads || !workers)
        return KVS_EINVAL;
    const PageChunks pc = pick_page_chunks(nres, n, num_layers, num_kv_heads, workers, parts_cap, extra_parts);
    *big = pc.big;
    *small = pc.small;
    *tail = pc.tail;
    return KVS_OK;
}

int kvs_debug_advance(kvs_ctx_t *ctx, uint64_t steps)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    ctx->t += steps;
    return KVS_OK;
}

int kvs_export_records(kvs_ctx_t *ctx, uint64_t seq_id, void *host_dst, size_t host_bytes, void *stream)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    uint32_t slot;
    SeqState *s = find_seq(ctx, seq_id, &slot);
    if (!s)
        return fail(ctx, KVS_ENOTFOUND, "unknown sequence %llu", (unsigned long long)seq_id);
    const size_t nb = s->table.size();
    const size_t want = nb * sizeof(kvs_record);
    const size_t n = std::min(want, host_bytes / sizeof(kvs_record) * sizeof(kvs_record));
    if (n) {
        CU(cudaMemcpyAsync(host_dst, static_cast<kvs_record *>(ctx->buf.records) + static_cast<size_t>(slot) * ctx->cfg.max_blocks_per_seq,
                           n, cudaMemcpyDeviceToHost, S(stream)));
        WAIT(S(stream));
    }
    if (n < want)
        return fail(ctx, KVS_ETRUNC, "host buffer holds %zu of %zu records", n / 64, nb);
    return KVS_OK;
}

int kvs_debug_import_records(kvs_ctx_t *ctx, uint64_t seq_id, const void *host_src, size_t host_bytes,
                             void *stream)
{
    KVS_RANGE();
    if (!ctx || !host_src)
        return KVS_EINVAL;
    uint32_t slot;
    SeqState *s = find_seq(ctx, seq_id, &slot);
    if (!s)
        return fail(ctx, KVS_ENOTFOUND, "unknown sequence %llu", (unsigned long long)seq_id);
    const size_t nb = s->table.size();
    if (host_bytes != nb * sizeof(kvs_record))
        return fail(ctx, KVS_EINVAL, "expected %zu records (%zu bytes), got %zu bytes", nb,
                    nb * sizeof(kvs_record), host_bytes);
    const kvs_record *src = static_cast<const kvs_record *>(host_src);
    for (size_t b = 0; b < nb; ++b)
        if (src[b].key.seq_id != seq_id || src[b].key.block_idx != b)
            return fail(ctx, KVS_EINVAL, "record %zu carries key (%llu, %llu)", b,
                        (unsigned long long)src[b].key.seq_id, (unsigned long long)src[b].key.block_idx);
    if (nb) {
        CU(cudaMemcpyAsync(static_cast<kvs_record *>(ctx->buf.records) + static_cast<size_t>(slot) * ctx->cfg.max_blocks_per_seq,
                           host_src, host_bytes, cudaMemcpyHostToDevice, S(stream)));
        WAIT(S(stream));
    }
    return KVS_OK;
}

int kvs_seq_info(kvs_ctx_t *ctx, uint64_t seq_id, uint32_t *slot, uint32_t *n_tokens,
                 uint32_t *n_blocks, int32_t *table_out, uint32_t table_cap)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    uint32_t sl;
    SeqState *s = find_seq(ctx, seq_id, &sl);
    if (!s)
        return fail(ctx, KVS_ENOTFOUND, "unknown sequence %llu", (unsigned long long)seq_id);
    if (slot)
        *slot = sl;
    if (n_tokens)
        *n_tokens = s->ntok;
    if (n_blocks)
        *n_blocks = static_cast<uint32_t>(s->table.size());
    if (table_out)
        for (uint32_t i = 0; i < table_cap && i < s->table.size(); ++i)
            table_out[i] = s->table[i];
    return KVS_OK;
}

int kvs_set_decode_events(kvs_ctx_t *ctx, void *ev_start, void *ev_stop)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    if ((ev_start == nullptr) != (ev_stop == nullptr))
        return fail(ctx, KVS_EINVAL, "give both events or neither");
    ctx->ev_dec_start = static_cast<cudaEvent_t>(ev_start);
    ctx->ev_dec_stop = static_cast<cudaEvent_t>(ev_stop);
    return KVS_OK;
}

int kvs_debug_inject(uint32_t faults, uint32_t wait_limit_ms)
{
    KVS_RANGE();
    if (faults & ~(KVS_FAULT_HOSTALLOC | KVS_FAULT_WAIT))
        return KVS_EINVAL;
    g_faults.store(faults);
    g_wait_limit_ms.store(wait_limit_ms ? wait_limit_ms : 600000u);
    return KVS_OK;
}

uint64_t kvs_kernel_launches(const kvs_ctx_t *ctx)
{
    KVS_RANGE();
    return ctx ? ctx->kernel_launches : 0;
}

uint64_t kvs_step_count(const kvs_ctx_t *ctx) { return ctx ? ctx->t : 0; }

uint32_t kvs_free_pages(const kvs_ctx_t *ctx)
{
    KVS_RANGE();
    return ctx ? static_cast<uint32_t>(pages_available(ctx)) : 0;
}

int kvs_check_device(kvs_ctx_t *ctx, void *stream)
{
    KVS_RANGE();
    if (!ctx)
        return KVS_EINVAL;
    cudaStream_t s = S(stream);
    CU(cudaMemcpyAsync(ctx->pinned_small, ctx->work.err, 8, cudaMemcpyDeviceToHost, s));
    WAIT(s);
    const uint32_t e = ctx->pinned_small[0], info = ctx->pinned_small[1];
    if (!e)
        return KVS_OK;
    CU(cudaMemsetAsync(ctx->work.err, 0, 8, s));
    WAIT(s);
    if (e & kErrTmaTimeout)
        return fail(ctx, KVS_ETIMEOUT, "a decode kernel gave up waiting for a TMA copy (error word 0x%x)", e);
    return fail(ctx, KVS_EDEVICE, "device error word 0x%x (bad page %d, bad record %d), info 0x%x", e,
                !!(e & kErrBadPage), !!(e & kErrBadRecord), info);
}

}  // extern "C"
