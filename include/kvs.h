/*
 * kvs.h -- C ABI of the paged KV-cache decode and block-scoring library
 * (one GPU, sm_103a).
 *
 * The library runs one hot path:
 *   append token K/V into 16-token pages reached through a per-sequence block
 *   table -> grouped-query decode attention over every cached token ->
 *   attention mass per (sequence, block), aggregated over all (layer, KV head)
 *   streams -> EMA/LRFU score, touch count and touch time in a 64-byte record
 *   per block -> priority P and tier -> selection of low-priority blocks ->
 *   gather of their pages into a pinned-host staging buffer -> identity-keyed
 *   re-admission that restores the record instead of resetting it.
 *
 * Sources, cited by page title and section:
 *   [VA]   "KV-Cache Offloading for LLM Inference -- Visual Reference" (v6.0):
 *          s.1 model geometry, s.3 KV size formula, s.4 decode reads the whole
 *          KV cache, s.11 EMA update rule, s.12 priority formula and tier
 *          thresholds (Diagrams 12.1, 12.2).
 *   [GQA]  "GQA per-head attention as scoring streams" figure page: 64 query
 *          heads grouped 8:1 onto 8 KV heads, 640 (layer, KV head) streams
 *          aggregated into one score per (sequence, 16-token block), the
 *          64-byte per-block state, identity-keyed persistence across
 *          eviction.
 *   [ARCH] "LLM KV cache offload" architecture page: block manager with
 *          fixed-size blocks and per-sequence block tables, reference counts
 *          for shared prefixes, eviction by demotion through pinned host
 *          staging on the copy engines, contiguous block layout.
 *   [RETR] "RETRACTIONS" page, s.2: blocks are write-once.
 *
 * Conventions for every call:
 *   - Status: every function returns KVS_OK (0) or a kvs_status code;
 *     kvs_last_error() then describes the failure.  On failure no state of
 *     the context has changed unless the description says so.
 *   - Memory: the library allocates no device memory.  The caller allocates
 *     every device buffer (sizes from kvs_required_sizes) and keeps it alive
 *     until kvs_destroy.  Host buffers passed to the gather/readmit calls are
 *     caller-owned pinned memory (cudaHostAlloc).  The context itself owns
 *     only host bookkeeping, CUDA events and a small pinned upload ring.
 *   - Streams: `stream` arguments are cudaStream_t values passed as void*.
 *     Calls are stream-ordered and asynchronous unless documented as
 *     synchronising: device outputs are valid once the stream has reached
 *     the call.  Calls on one context must be ordered by the caller (one
 *     stream, or events between streams).
 *   - Layouts (bf16 = IEEE bfloat16, little-endian):
 *       page   : [L][2 (K, V)][Hkv][16 token slots][d] elements, page_bytes =
 *                2*L*Hkv*16*d*elem (5,242,880 B for 80/8/128 in bf16); slots
 *                past the last token of a partial block are zero.  An element
 *                is a bf16 value, or with kv_dtype KVS_KV_FP8_E4M3 one byte
 *                holding an FP8 E4M3 code (page 2,621,440 B).
 *       pool   : [pool_blocks] pages.
 *       q      : [nseq][L][Hq][d] bf16; out: [nseq][L][Hq][d] float32.
 *       K, V   : token-major [n][L][Hkv][d] bf16 (as produced by a layer's
 *                projections for n consecutive tokens).
 *       record : 64 bytes, see kvs_record.
 *       mass   : float32 [max_seqs][max_blocks_per_seq], row = sequence slot.
 */
#ifndef KVS_H
#define KVS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVS_BLOCK_TOKENS 16u
#define KVS_RECORD_BYTES 64u
#define KVS_MAX_CALL_SEQS 256u   /* sequences in one decode call */
#define KVS_PREFETCH_MAX 4096u   /* blocks in one prefetch plan */

/* Opaque context: host bookkeeping of one pool (free list, reference counts,
 * block tables, identity store), its events and its upload ring. */
typedef struct kvs_ctx kvs_ctx_t;

typedef enum kvs_status {
    KVS_OK = 0,
    KVS_EINVAL = 1,     /* bad argument or call in the wrong state */
    KVS_ENOMEM = 2,     /* pool pages, sequence slots or staging exhausted */
    KVS_ECUDA = 3,      /* a CUDA runtime call failed */
    KVS_ENOTFOUND = 4,  /* unknown sequence or identity key */
    KVS_EEXIST = 5,     /* sequence or key already present / resident */
    KVS_ETRUNC = 6,     /* output buffer too small: partial result written */
    KVS_ETIMEOUT = 7,   /* a bounded wait ran out (device or host) */
    KVS_EDEVICE = 8     /* a kernel reported an inconsistency (see error text) */
} kvs_status;

typedef enum kvs_kv_dtype {
    KVS_KV_BF16 = 0,       /* pages hold bf16 K and V                          */
    KVS_KV_FP8_E4M3 = 1,   /* pages hold FP8 E4M3 codes: value = code * scale,
                              appended bf16 values quantised as
                              code = e4m3(x / scale) ("Fitting a Million
                              Tokens", s.02: FP8 E4M3 KV halves the bytes)    */
    KVS_KV_KIVI2 = 2       /* 2-bit groups behind a bf16 residual window
                              ("Fitting a Million Tokens", s.02, KIVI): see
                              KVS_KIVI_* below                               */
} kvs_kv_dtype;

/* KIVI-style 2-bit KV (kv_dtype KVS_KV_KIVI2, head_dim 128).  Pages are
 * written in bf16 as usual; once a sequence holds n tokens, every whole group
 * of 32 tokens (two blocks) that ends at least 128 tokens before the end --
 * the first 32*floor(max(0, n-128)/32) tokens -- is quantised into a group
 * page and its two bf16 pages go back to the free list.  Keys: per channel
 * over the group's 32 tokens; values: per token over groups of 32 channels;
 * asymmetric 2-bit, in fp32: mn, mx = min, max; scale = fp16((mx-mn)/3);
 * zero = fp16(mn); code = clamp(rint((x - zero)/scale), 0, 3) (ties to even;
 * 0 when scale is 0).  Attention reads fp16(code*scale + zero) (one
 * rounding).  A group page holds, per (layer, KV head), 3072 bytes: K codes,
 * V codes, K (scale, zero) per channel, V (scale, zero) per token and channel
 * group, each scale stored doubled (exact in fp16) -- 3 bits per element.  The table entry of a quantised block is
 * KVS_TABLE_GROUP(g) for its group page g (both blocks of the group).
 * KIVI contexts share no blocks between sequences and gather no pages
 * (kvs_select_and_gather returns the id list only: no host_dst, flags 0 or
 * KVS_GATHER_ASYNC). */
#define KVS_KIVI_GROUP_TOKENS 32u
#define KVS_KIVI_RESIDUAL 128u
#define KVS_KIVI_TILE_BYTES 3072u
#define KVS_TABLE_GROUP(g) (-2 - (int32_t)(g))

typedef enum kvs_select_mode {
    KVS_SELECT_THRESH = 0,   /* every record with P < cut_lo (tier 2) */
    KVS_SELECT_LOWFRAC = 1,  /* the floor(frac*N) records with smallest P */
    KVS_SELECT_LRFU = 2      /* the floor(frac*N) records with smallest LRFU key */
} kvs_select_mode;

/* kvs_gather_args.flags */
#define KVS_GATHER_DEMOTE 1u  /* free the gathered pages, keep records by key */
#define KVS_GATHER_MIRROR 2u  /* host_dst mirrors the pool (page p at p*page_bytes);
                                 pages whose host copy is current are not re-sent */
#define KVS_GATHER_ASYNC 4u   /* with MIRROR, or alone in a 2-bit context: no host
                                 wait; counts later from kvs_gather_counts */

typedef struct kvs_config {
    uint32_t num_layers;          /* L                                        */
    uint32_t num_q_heads;         /* Hq                                       */
    uint32_t num_kv_heads;        /* Hkv; Hq % Hkv == 0, Hq/Hkv <= 8          */
    uint32_t head_dim;            /* d: 64 or 128                             */
    uint32_t block_tokens;        /* must be 16                               */
    uint32_t pool_blocks;         /* physical pages in the pool               */
    uint32_t max_seqs;            /* sequence slots                           */
    uint32_t max_blocks_per_seq;  /* block-table row length                   */
    uint32_t max_call_blocks;     /* max sum of blocks over one decode call;
                                     0 = max_seqs * max_blocks_per_seq       */
    uint32_t staging_pages;       /* device staging ring, pages (>= 1)        */
    double alpha;                 /* EMA weight of the current mass [VA] s.11 */
    uint32_t recency_window;      /* W: R = clip(1 - (t - last_touch)/W, 0, 1) */
    uint32_t kv_dtype;            /* kvs_kv_dtype; FP8 needs head_dim 128     */
    double w_recency, w_ema, w_anchor;   /* [VA] s.12: 0.25, 0.55, 0.20      */
    double cut_lo, cut_hi;               /* [VA] Diagram 12.2: 0.3, 0.6      */
    uint64_t pool_seed;           /* seeds the free-list order of the pool    */
    float k_scale, v_scale;       /* FP8 only: per-tensor scales (> 0); the
                                     quotient x / scale is an IEEE fp32
                                     division, rounded to the nearest code
                                     (ties to even), saturating at +-448   */
    uint32_t kivi_groups;         /* KIVI only: group pages in the group pool */
    uint32_t reserved1;           /* 0                                        */
} kvs_config;

/* Byte sizes of the caller-allocated device buffers.  Every buffer must be
 * 256-byte aligned (cudaMalloc and the PyTorch caching allocator are). */
typedef struct kvs_sizes {
    size_t page_bytes;
    size_t pool_bytes;        /* pool_blocks * page_bytes                     */
    size_t table_bytes;       /* int32 [max_seqs][max_blocks_per_seq]         */
    size_t records_bytes;     /* kvs_record [max_seqs][max_blocks_per_seq]    */
    size_t mass_bytes;        /* float [max_seqs][max_blocks_per_seq]         */
    size_t workspace_bytes;   /* decode partials, per-block LSE, select state */
    size_t staging_bytes;     /* staging_pages * page_bytes                   */
    size_t group_page_bytes;  /* KIVI: L * Hkv * KVS_KIVI_TILE_BYTES, else 0  */
    size_t group_pool_bytes;  /* KIVI: kivi_groups * group_page_bytes, else 0 */
} kvs_sizes;

typedef struct kvs_buffers {
    void *pool, *block_table, *records, *mass, *workspace, *staging;
    void *group_pool;         /* KIVI only (group_pool_bytes), else NULL      */
} kvs_buffers;

/* Identity key of a block [GQA]: the sequence it belongs to and its logical
 * block index.  16 bytes. */
typedef struct kvs_key {
    uint64_t seq_id;
    uint64_t block_idx;
} kvs_key;

/* The 64-byte per-block state [GQA]: 16 B identity key, 8 B score, 8 B touch
 * timestamp, 4 B touch count, then reserved bytes, which hold the tier, the
 * last priority, the last mass and the event-driven (LRFU) score. */
typedef struct kvs_record {
    kvs_key key;          /*  0 */
    double score;         /* 16  EMA of the block mass, 0 at creation        */
    uint64_t last_touch;  /* 24  step of the last touch (creation step first) */
    uint32_t count;       /* 32  touches so far                              */
    uint8_t tier;         /* 36  0, 1, 2; 255 = not scored yet               */
    uint8_t flags;        /* 37  bit 0: demoted (not resident)               */
    uint16_t pad0;        /* 38                                              */
    double prio;          /* 40  last P                                      */
    float mass;           /* 48  last block mass M                           */
    uint8_t reserved[4];  /* 52                                              */
    double lrfu;          /* 56  event-driven score right after the last
                           *     touch (0 if never touched), [RETR] s.3      */
} kvs_record;

typedef struct kvs_gather_args {
    int32_t mode;            /* kvs_select_mode                                */
    uint32_t flags;          /* KVS_GATHER_*                                   */
    double frac;             /* LOWFRAC fraction of all records (e.g. 0.10)    */
    void *host_dst;          /* pinned host buffer, caller-owned               */
    size_t host_dst_bytes;
    kvs_key *ids_dev;        /* device out [ids_capacity]: selected keys in list
                                order (may be NULL)                            */
    int32_t *slot_dev;       /* device out [ids_capacity]: page index in host_dst
                                holding each id's bytes, -1 if not gathered
                                (may be NULL)                                  */
    uint32_t ids_capacity;
    uint32_t reserved0;
    void *stream;            /* main stream (selection, gather kernels)       */
    void *side_stream;       /* copy stream for device->host (may == stream)  */
} kvs_gather_args;

typedef struct kvs_gather_result {
    uint32_t n_selected;     /* records in the list                           */
    uint32_t n_pages;        /* pages the list makes eligible (deduplicated)  */
    uint32_t n_staged;       /* pages written to host_dst by this call        */
    uint32_t n_demoted;      /* records demoted (KVS_GATHER_DEMOTE)           */
    uint64_t bytes_to_host;  /* bytes copied device -> host by this call      */
} kvs_gather_result;

/* Sizes of every caller-allocated device buffer for `cfg`.
 * Returns KVS_EINVAL (with no sizes) if cfg is not supported. */
int kvs_required_sizes(const kvs_config *cfg, kvs_sizes *out);

/* Creates a context over caller-allocated device buffers (sizes from
 * kvs_required_sizes, all on the current device): the block manager of
 * [ARCH] -- a pool of fixed-size blocks handed out from a free list, a
 * block table per sequence, reference counts for shared blocks -- whose
 * bookkeeping the context holds on the host.  Zeroes the block table,
 * records and mass (synchronously) and builds the pool's TMA descriptor.
 * The free list holds every pool page in an order seeded by cfg->pool_seed. */
int kvs_create(const kvs_config *cfg, const kvs_buffers *buf, kvs_ctx_t **out);

/* Destroys host state and events; does not touch caller buffers.  Waits for
 * work the context enqueued. */
void kvs_destroy(kvs_ctx_t *ctx);

/* Text of the last failure on this context (owned by the context).  With
 * ctx NULL: the last failure of a call made without a context
 * (kvs_required_sizes, a failed kvs_create) on the calling thread. */
const char *kvs_last_error(const kvs_ctx_t *ctx);

/* Adds a sequence with no tokens.  With parent_seq_id >= 0, the first
 * shared_prefix_blocks (full) blocks of the parent are shared read-only:
 * the new table points at the same pages and their reference counts rise
 * [ARCH]; the new sequence gets its own records for those blocks (score 0,
 * count 0, last_touch = current step), written on `stream`.  Appending
 * never writes a shared page.  KVS_EEXIST if seq_id is
 * present, KVS_ENOTFOUND if the parent is not, KVS_ENOMEM if no slot is
 * free, KVS_EINVAL if the parent has fewer full blocks or, in a 2-bit
 * (KVS_KV_KIVI2) context, if any block is to be shared. */
int kvs_seq_add(kvs_ctx_t *ctx, uint64_t seq_id, int64_t parent_seq_id,
                uint32_t shared_prefix_blocks, void *stream);

/* Removes a sequence: its pages lose one reference each and return to the
 * free list at zero; its 2-bit group pages return to the group free list;
 * its demoted keys are dropped.  Stream-ordered after `stream` (page reuse
 * waits for work enqueued before). */
int kvs_seq_remove(kvs_ctx_t *ctx, uint64_t seq_id, void *stream);

/* Appends n tokens to a sequence [ARCH]: K and V are device, token-major
 * [n][L][Hkv][d] bf16.  A page is taken from the free list whenever a token
 * opens a new block; the page's later slots are zero-filled and the block's
 * record is created with score 0, count 0, last_touch = the current step
 * counter (decode steps completed so far), tier 255.  In a 2-bit context the
 * groups that fall behind the residual window are then quantised into group
 * pages on `stream` and their bf16 pages freed (KVS_KV_KIVI2 above).
 * KVS_ENOMEM if the free list (or the group pool) runs out (nothing
 * appended), KVS_EINVAL for n == 0 or a table row overflow. */
int kvs_append_tokens(kvs_ctx_t *ctx, uint64_t seq_id, uint32_t n,
                      const void *k_dev, const void *v_dev, void *stream);
int kvs_append_token(kvs_ctx_t *ctx, uint64_t seq_id, const void *k_dev,
                     const void *v_dev, void *stream);

/* Appends one token to each of nseq sequences in one launch (the new K/V rows
 * of a decode step) [ARCH]: k, v device [nseq][L][Hkv][d] bf16, row i for
 * seq_ids[i].  Same effect as kvs_append_token for each sequence in turn:
 * a token that opens a block takes a page from the free list (tail slots
 * zeroed, record created with the current step counter), and in a 2-bit
 * context the groups that become due are quantised in one launch.
 * KVS_ENOMEM if the free list (or the group pool) cannot cover every new
 * block (nothing appended); KVS_EINVAL for duplicates, a full table row, or
 * a last block that is shared or demoted. */
int kvs_append_step(kvs_ctx_t *ctx, const uint64_t *seq_ids, uint32_t nseq,
                    const void *k_dev, const void *v_dev, void *stream);

/* One decode step for nseq sequences [VA] s.4, [GQA]: advances the step
 * counter t by one, then for every (sequence, layer, query head) computes
 *   out = sum_t softmax_t(q.k_t / sqrt(d)) v_t   over all cached tokens,
 * (query head h reads KV head h / (Hq/Hkv)), and for every block b of each
 * sequence the aggregated mass
 *   M(b) = 1/(L*Hq) * sum_{l,h} sum_{t in b} softmax weight,
 * written to mass[slot][b].  q [nseq][L][Hq][d] bf16 and out [nseq][L][Hq][d]
 * float32 are device, in the order of seq_ids.  The set of sequences becomes
 * the one kvs_score_update and kvs_select_and_gather work on.  In a 2-bit
 * context the blocks in group pages are read through one kernel and the
 * residual pages through the page kernel; both feed the same merge.
 * KVS_EINVAL: nseq == 0 or > KVS_MAX_CALL_SEQS, duplicates, an empty
 * sequence or one with a demoted block; KVS_ENOTFOUND: unknown id. */
int kvs_decode_step(kvs_ctx_t *ctx, const uint64_t *seq_ids, uint32_t nseq,
                    const void *q_dev, float *out_dev, void *stream);

/* kvs_decode_step followed by kvs_score_update, in fewer launches: the
 * epilogue that writes each block's mass scores the block's record in the
 * same kernel ([GQA]: the aggregated mass lands in the 64-byte record).
 * Results are bit-identical to the two calls.  kvs_score_update must not be
 * called for a set this call scored (KVS_EINVAL).  Errors as
 * kvs_decode_step. */
int kvs_decode_score_step(kvs_ctx_t *ctx, const uint64_t *seq_ids, uint32_t nseq,
                          const void *q_dev, float *out_dev, void *stream);

/* Scores every block of the last decode set [VA] s.11, s.12, [GQA]:
 *   E <- alpha*M + (1-alpha)*E;  if M*num_blocks >= 1 (a touch):
 *   count += 1, lrfu <- alpha + (1-alpha)^(t - last_touch) * lrfu,
 *   last_touch = t;  R = clip(1 - (t - last_touch)/W, 0, 1);
 *   N = 1 for block 0 and the newest block, else 0;
 *   P = w_recency*R + w_ema*E + w_anchor*N;
 *   tier = 0 if P >= cut_hi, 1 if cut_lo <= P < cut_hi, 2 if P < cut_lo.
 * fp64 with no fused multiply-add, in that order.  lrfu is the EMA of the
 * touch indicator, decayed lazily ([RETR] s.3): its value at any step t is
 * lrfu * (1-alpha)^(t - last_touch); the power is taken by binary
 * exponentiation (result = 1, base = 1-alpha; per bit of the exponent from
 * the lowest: if set result *= base; base *= base). */
int kvs_score_update(kvs_ctx_t *ctx, void *stream);
/* (KVS_EINVAL if the last set was already scored by kvs_decode_score_step.) */

/* Changes alpha for later score updates. */
int kvs_set_alpha(kvs_ctx_t *ctx, double alpha);

/* Selects records of the last decode set and gathers their pages
 * [VA] s.12, [ARCH].  Synchronising: returns after the list is known and
 * every copy is enqueued; host_dst is complete once args->side_stream has
 * reached this call.
 *   THRESH : every record with tier 2, ascending (seq_id, block_idx).
 *   LOWFRAC: the floor(frac*N) records of smallest (P, seq_id, block_idx)
 *            over all N records of the set, listed ascending (seq_id,
 *            block_idx).
 *   LRFU   : as LOWFRAC with the order-preserving key of [RETR] s.3,
 *            K = ln(lrfu) + last_touch * (-ln(1 - alpha)) (-inf when lrfu
 *            is 0), in place of P: the records whose lazily decayed LRFU
 *            score is smallest at any step.  Both logarithms come from the
 *            series ln x = e ln2 + 2 artanh(s), x = m 2^e with m in
 *            [sqrt(1/2), sqrt(2)), s = (m-1)/(m+1), the odd powers of s up
 *            to s^23 by Horner's rule, each step one round-to-nearest fp64
 *            operation in that order (no fused multiply-add), so that keys
 *            and their order are reproducible bit for bit off the device.
 *            KVS_EINVAL if alpha >= 1.
 * A page is eligible when every record that references it is in the list
 * (a shared page is released only by its last user); each eligible page is
 * gathered once, at the position of its first record.  Default: eligible
 * pages go into host_dst in list order through the device staging ring;
 * if host_dst is too small a prefix is written and KVS_ETRUNC returned with
 * the full counts.  KVS_GATHER_MIRROR: host_dst holds pool_blocks pages and
 * page p goes to offset p*page_bytes; a page whose host copy is still
 * current (written whole and unchanged since, [RETR] s.2) is not copied
 * again.  KVS_GATHER_DEMOTE (list mode only): eligible records are demoted:
 * their 64-byte record and the offset of their page in host_dst are kept
 * under their key, the table entry is cleared and the page freed.  The
 * caller keeps host_dst alive until kvs_readmit.
 * KVS_GATHER_ASYNC (with KVS_GATHER_MIRROR, or as the only flag of a 2-bit
 * context): the call enqueues its work on `stream` and returns without
 * waiting for the device; *res is zeroed.  The stale pages are written into
 * host_dst by a device kernel on `stream` through the buffer's device
 * mapping, so host_dst must be page-locked memory the device can address
 * (cudaHostAlloc / cudaMallocHost, or cudaHostRegister'ed): KVS_EINVAL
 * otherwise.  ids_dev and slot_dev receive min(ids_capacity, N) entries;
 * those past the list's length are unspecified.  The counts of the latest
 * such call come from kvs_gather_counts.  KVS_EINVAL with DEMOTE or in list
 * mode. */
int kvs_select_and_gather(kvs_ctx_t *ctx, const kvs_gather_args *args,
                          kvs_gather_result *res);

/* Counts of the latest KVS_GATHER_ASYNC select: waits (bounded, KVS_ETIMEOUT)
 * until that call's work on its stream has reached them -- with MIRROR, until
 * its page copies are visible in the host mirror -- then fills *res as a
 * synchronous call would have (n_demoted = 0).  A MIRROR call signals this
 * through a pinned word its last kernel writes, not through a stream event,
 * so that nothing in the stream separates it from the next kernels; the
 * stream must stay alive until the counts are read.  KVS_ECUDA if the stream
 * fails meanwhile, KVS_EDEVICE if it drains without the signal.  KVS_EINVAL
 * if no asynchronous select was made on this context. */
int kvs_gather_counts(kvs_ctx_t *ctx, kvs_gather_result *res);

/* Re-admits demoted blocks [GQA]: for each key, takes a page from the free
 * list, copies the page bytes from host_src (the buffer given to the demoting
 * gather) and restores the 64-byte record bit for bit.  KVS_ENOTFOUND for a
 * key that is not demoted, KVS_EEXIST for a duplicate key in `keys`,
 * KVS_ENOMEM if the free list runs out (nothing re-admitted). */
int kvs_readmit(kvs_ctx_t *ctx, const kvs_key *keys, uint32_t n,
                const void *host_src, size_t host_src_bytes, void *stream);

/* Fetch order of the demoted blocks, [VA] s.14 "Prefetching Strategy"
 * (Diagram 14.1 targets, in order: the anchor zone, token positions 0..100;
 * the recent window, positions m-200..m-1 where m is the sequence's token
 * count; high-EMA blocks) with the fetch priority 1/(1 + distance/100) and
 * the fetch-order blend 0.6 rope_factor + 0.4 ema_factor named beside the
 * [VA] s.12 priority formula.  For every demoted block of a live sequence
 * the device computes
 *   class = 0 if the block holds a position <= 100, else 1 if it holds a
 *           position >= m - 200, else 2;
 *   distance = max(0, (m - 1) - (16*block_idx + 15));
 *   blend = min(1, 0.6 * (1 / (1 + distance/100)) + 0.4 * E)
 * (fp64, each operation rounded in that order, no fused multiply-add; E is
 * the record's EMA score kept since demotion) and orders the blocks by
 * (class ascending, blend descending, seq_id ascending, block_idx
 * ascending).  The first n = min(budget, demoted) entries are written to
 * keys_out[n] and, if given, blend_out[n] and class_out[n] (all host).
 * Synchronising on `stream`.  KVS_EINVAL: budget > KVS_PREFETCH_MAX or a
 * missing output.  n_out = 0 when nothing is demoted. */
int kvs_prefetch_plan(kvs_ctx_t *ctx, uint32_t budget, kvs_key *keys_out,
                      double *blend_out, uint8_t *class_out, uint32_t *n_out,
                      void *stream);

/* kvs_prefetch_plan, then kvs_readmit of those blocks with their
 * host-to-device copies issued in plan order (highest priority first) on
 * `stream`; pass a stream other than the one decoding so that the copies
 * run on a copy engine beside the decode kernels.  The re-admitted blocks
 * are in place once `stream` reaches the end of this call: make the
 * decoding stream wait for it (an event) before it decodes their
 * sequences.  host_src and the errors are those of kvs_readmit (nothing is
 * re-admitted on an error). */
int kvs_prefetch(kvs_ctx_t *ctx, uint32_t budget, const void *host_src,
                 size_t host_src_bytes, kvs_key *keys_out, double *blend_out,
                 uint8_t *class_out, uint32_t *n_out, void *stream);

/* Test hook: makes seq_ids the current set and copies mass_dev (float32
 * [nseq][max_blocks_per_seq], row i for seq_ids[i], device) into the mass
 * rows, without decoding and without advancing t.  Lets the scoring,
 * tiering and selection steps be driven from given masses. */
int kvs_debug_set_mass(kvs_ctx_t *ctx, const uint64_t *seq_ids, uint32_t nseq,
                       const float *mass_dev, void *stream);

/* Test hook: advances the step counter without decoding. */
int kvs_debug_advance(kvs_ctx_t *ctx, uint64_t steps);

/* Copies the records of one sequence (block order, 64 B each) to host_dst.
 * Synchronising.  KVS_ETRUNC if host_bytes holds fewer than all blocks. */
int kvs_export_records(kvs_ctx_t *ctx, uint64_t seq_id, void *host_dst,
                       size_t host_bytes, void *stream);

/* Test hook (the pages have no counterpart): overwrites the records of one
 * sequence with host_src (block order, 64 B each, exactly all its blocks),
 * so that selection can be driven from planted records.  Every record must
 * carry the sequence's key (seq_id, block index): KVS_EINVAL otherwise, and
 * for a size other than 64 * blocks.  Synchronising. */
int kvs_debug_import_records(kvs_ctx_t *ctx, uint64_t seq_id, const void *host_src,
                             size_t host_bytes, void *stream);

/* Host view of a sequence: its slot (row of the table, records and mass
 * buffers), token count, block count, and (if table_out is not NULL) up to
 * table_cap page ids (-1 = demoted, KVS_TABLE_GROUP(g) = held in 2-bit group
 * page g).  Any output pointer may be NULL. */
int kvs_seq_info(kvs_ctx_t *ctx, uint64_t seq_id, uint32_t *slot,
                 uint32_t *n_tokens, uint32_t *n_blocks, int32_t *table_out,
                 uint32_t table_cap);

/* Measurement hook: when ev_start/ev_stop (cudaEvent_t as void*) are not
 * NULL, every later kvs_decode_step records ev_start on its stream right
 * before the split-K decode kernel(s) and ev_stop right after, so they can
 * be timed on the stream they run on (2-bit contexts: both launches).  NULL, NULL turns it off.  The
 * events stay owned by the caller. */
int kvs_set_decode_events(kvs_ctx_t *ctx, void *ev_start, void *ev_stop);

/* Decode attention and per-block mass of ONE sequence, for callers that
 * cannot allocate device memory.  The pages have no counterpart for this
 * call: it exists for programs that are handed only their input and output
 * buffers -- a plugin or custom operator running inside another framework's
 * memory budget, or a serving loop that forbids allocation after start-up.
 *
 * Same arithmetic as kvs_decode_step (same kernels) for one sequence, with no
 * context: pool ([pool_blocks] pages, layout as above), block_table (int32,
 * ceil(n_tokens/16) page ids), q [L][Hq][d] bf16 and outputs out [L][Hq][d]
 * float32 and mass [ceil(n_tokens/16)] float32, all device memory owned by
 * the caller.  The decode scratch lives in a fixed 48 MiB array compiled into
 * the library (held by every GPU that loads it, until exit); a call needing
 * more returns KVS_EINVAL with the required size in msg (for the 80-layer,
 * 8-KV-head, d=128 shape the limit is 12,288 tokens).  Nothing is allocated:
 * no cudaMalloc, cudaFree or allocating library routine.
 *
 * status (optional, device, 2 x uint32, 4-byte aligned, caller-owned):
 * written in stream order after the outputs with the kernels' error word
 * (bit 0: a block-table entry outside [0, pool_blocks) -- demoted or 2-bit
 * entries included -- was read; the kernel used page 0 in its place, so out
 * and mass are not valid; bit 1: a wait for a TMA copy ran out) and the
 * first offending table value or-ed with 0x80000000 (0: none).  {0, 0}:
 * out and mass are valid.  With
 * status NULL such a problem goes unreported (the call still returns KVS_OK
 * once its work is enqueued).
 *
 * The first call on a device (with that device current) looks up the array's
 * device address and the decode kernel's occupancy; make that first call
 * before any stream capture.  Every call shares the array: calls that overlap
 * on the GPU race, so order them (one stream).  The array keeps the last
 * call's contents; what must start at zero is cleared by each call.
 * msg (optional, msg_bytes long) receives a description of a failure. */
int kvs_decode_noalloc(uint32_t num_layers, uint32_t num_q_heads,
                       uint32_t num_kv_heads, uint32_t head_dim,
                       const void *pool, uint32_t pool_blocks,
                       const int32_t *block_table, uint32_t n_tokens,
                       const void *q, float *out, float *mass, uint32_t *status,
                       void *stream, char *msg, size_t msg_bytes);

/* Test hook, process-wide (the pages have no counterpart): injects host-side
 * failures so that error paths can be exercised without a GPU fault.
 *   KVS_FAULT_HOSTALLOC: the pinned host allocation of the next kvs_create
 *                        fails (KVS_ENOMEM; one shot; nothing leaks);
 *   KVS_FAULT_WAIT:      every host wait of the library (read-backs, upload
 *                        ring, kvs_check_device) sees its event as not yet
 *                        complete, so it ends with KVS_ETIMEOUT after
 *                        wait_limit_ms (the device work stays enqueued).
 * wait_limit_ms also sets the limit of real waits (0 = 600,000 ms, the
 * default).  kvs_debug_inject(0, 0) clears everything.  KVS_EINVAL for
 * unknown bits. */
#define KVS_FAULT_HOSTALLOC 1u
#define KVS_FAULT_WAIT 2u
int kvs_debug_inject(uint32_t faults, uint32_t wait_limit_ms);

/* Test hook, process-wide, no GPU needed (the pages have no counterpart): the
 * decode work-item plan the library uses for one call.  Sequence i of the n
 * has nres[i] blocks in each of its num_layers x num_kv_heads streams;
 * `workers` decode warps claim the items; at most parts_cap chunk partials
 * may be used, extra_parts of them already taken.  A stream of m blocks is
 * cut into nbig = (m > tail ? (m - tail) / big : 0) chunks of `big` blocks
 * followed by chunks of `small` blocks (the last one shorter), claimed
 * chunk by chunk.  *big = 0 when no plan fits parts_cap.  KVS_EINVAL for
 * null pointers, n == 0, or zero layers, heads or workers. */
int kvs_debug_chunk_plan(const uint32_t *nres, uint32_t n, uint32_t num_layers,
                         uint32_t num_kv_heads, uint32_t workers, uint64_t parts_cap,
                         uint64_t extra_parts, uint32_t *big, uint32_t *small,
                         uint32_t *tail);

/* Kernels this context has launched so far (every kernel of the library,
 * counted at launch). */
uint64_t kvs_kernel_launches(const kvs_ctx_t *ctx);

/* Decode steps completed so far (the step counter t). */
uint64_t kvs_step_count(const kvs_ctx_t *ctx);

/* Free pages left in the pool. */
uint32_t kvs_free_pages(const kvs_ctx_t *ctx);

/* Reads and clears the device error word (synchronising on `stream`).
 * KVS_OK if no kernel reported a problem, else KVS_EDEVICE / KVS_ETIMEOUT
 * with the description in kvs_last_error. */
int kvs_check_device(kvs_ctx_t *ctx, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* KVS_H */
