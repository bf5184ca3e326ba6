// Scoring of one block record from its mass, shared by the scoring kernel
// and the decode epilogue that scores as it writes the masses.  Not part of
// the public ABI.
//
// Sources: "KV-Cache Offloading for LLM Inference -- Visual Reference" s.11
// (E <- alpha*M + (1 - alpha)*E), s.12 (P = 0.25 R + 0.55 E + 0.20 N, tiers at
// P = 0.3 / 0.6); "GQA per-head attention as scoring streams" (the 64-byte
// record: key, score, touch time, touch count); "RETRACTIONS" s.3 (the
// lazily decayed event-driven score).
#pragma once

#include "kvs_internal.h"

namespace kvs {

// (1 - alpha)^dt by binary exponentiation: result = 1, base = 1 - alpha; per
// bit of dt from the lowest, if set result *= base; then base *= base.
__device__ __forceinline__ double lrfu_decay(double alpha, uint64_t dt)
{
    double base = __dsub_rn(1.0, alpha), res = 1.0;
    for (; dt; dt >>= 1) {
        if (dt & 1u)
            res = __dmul_rn(res, base);
        base = __dmul_rn(base, base);
    }
    return res;
}

// Scores block b of a sequence from its fp32 mass M at step t: rec is its
// record as loaded, dst where the scored record goes.  fp64, every operation
// rounded on its own (no fused multiply-add), in the order EMA, touch,
// recency, anchor, P, tier.  nb: the sequence's block count.  A record that
// does not carry (seq_id, b) or whose touch time lies after t is left alone
// and flagged in the error word.
//
// Split in two so that a kernel can take everything that does not depend on M
// (the record is final before M is): score_prep computes the mass-free terms
// -- (1 - alpha)*E, the touched record's decayed event score, the recency
// term for both outcomes of the touch test, the anchor term -- and
// score_finish the rest.  Each value is the same operation on the same
// operands as in the one-pass order above, so the record comes out bit for
// bit the same.
struct ScorePrep {
    double e_keep;      // (1 - alpha) * E
    double lrfu_touch;  // alpha + (1 - alpha)^(t - last touch) * lrfu: the event score if touched
    double rr_keep;     // wR * R, R from the age since the last touch (not touched)
    double rr_touch;    // wR * R, R from age 0 (touched at t)
    double nn;          // wN * N
    bool bad;           // key or touch time inconsistent: leave the record alone
};

__device__ __forceinline__ double recency_term(const ScoreArgs &sa, uint64_t age)
{
    double R = __dsub_rn(1.0, __ddiv_rn(static_cast<double>(age), static_cast<double>(sa.W)));
    R = fmin(fmax(R, 0.0), 1.0);
    return __dmul_rn(sa.wR, R);
}

__device__ __forceinline__ ScorePrep score_prep(const ScoreArgs &sa, const kvs_record &rec, uint64_t seq_id,
                                                uint32_t b, uint32_t nb, uint64_t t)
{
    ScorePrep p;
    p.bad = rec.key.block_idx != b || rec.key.seq_id != seq_id || rec.last_touch > t;
    if (p.bad) {
        p.e_keep = p.lrfu_touch = p.rr_keep = p.rr_touch = p.nn = 0.0;
        return p;
    }
    // E <- alpha*M + (1 - alpha)*E: the second product
    p.e_keep = __dmul_rn(__dsub_rn(1.0, sa.alpha), rec.score);
    // on a touch the event-driven score decays lazily from the previous touch
    p.lrfu_touch = __dadd_rn(sa.alpha, __dmul_rn(lrfu_decay(sa.alpha, t - rec.last_touch), rec.lrfu));
    p.rr_keep = recency_term(sa, t - rec.last_touch);
    p.rr_touch = recency_term(sa, 0);
    const double N = (b == 0 || b + 1 == nb) ? 1.0 : 0.0;
    p.nn = __dmul_rn(sa.wN, N);
    return p;
}

__device__ __forceinline__ void score_finish(const ScoreArgs &sa, const ScorePrep &p, kvs_record rec,
                                             kvs_record *dst, uint32_t nb, uint64_t t, float mass, uint32_t *err)
{
    if (p.bad) {
        atomicOr(err, kErrBadRecord);
        return;
    }
    const double M = static_cast<double>(mass);
    const double E = __dadd_rn(__dmul_rn(sa.alpha, M), p.e_keep);
    // touch: mass at or above the uniform share 1/num_blocks
    const bool touch = __dmul_rn(M, static_cast<double>(nb)) >= 1.0;
    if (touch) {
        rec.count += 1;
        rec.lrfu = p.lrfu_touch;
        rec.last_touch = t;
    }
    const double P = __dadd_rn(__dadd_rn(touch ? p.rr_touch : p.rr_keep, __dmul_rn(sa.wE, E)), p.nn);
    rec.score = E;
    rec.prio = P;
    rec.tier = P >= sa.hi ? 0 : (P >= sa.lo ? 1 : 2);
    rec.mass = mass;
    *dst = rec;
}

__device__ __forceinline__ void score_loaded(const ScoreArgs &sa, const kvs_record &rec, kvs_record *dst,
                                             uint64_t seq_id, uint32_t b, uint32_t nb, uint64_t t, float mass,
                                             uint32_t *err)
{
    score_finish(sa, score_prep(sa, rec, seq_id, b, nb, t), rec, dst, nb, t, mass, err);
}

__device__ __forceinline__ void score_record(const ScoreArgs &sa, kvs_record *recs, size_t idx, uint64_t seq_id,
                                             uint32_t b, uint32_t nb, uint64_t t, float mass, uint32_t *err)
{
    score_loaded(sa, recs[idx], recs + idx, seq_id, b, nb, t, mass, err);
}

}  // namespace kvs
