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
__device__ __forceinline__ void score_loaded(const ScoreArgs &sa, kvs_record rec, kvs_record *dst, uint64_t seq_id,
                                             uint32_t b, uint32_t nb, uint64_t t, float mass, uint32_t *err)
{
    if (rec.key.block_idx != b || rec.key.seq_id != seq_id || rec.last_touch > t) {
        atomicOr(err, kErrBadRecord);
        return;
    }
    const double M = static_cast<double>(mass);
    // E <- alpha*M + (1 - alpha)*E
    const double E = __dadd_rn(__dmul_rn(sa.alpha, M), __dmul_rn(__dsub_rn(1.0, sa.alpha), rec.score));
    // touch: mass at or above the uniform share 1/num_blocks; the
    // event-driven score decays lazily from the previous touch
    if (__dmul_rn(M, static_cast<double>(nb)) >= 1.0) {
        rec.count += 1;
        rec.lrfu = __dadd_rn(sa.alpha, __dmul_rn(lrfu_decay(sa.alpha, t - rec.last_touch), rec.lrfu));
        rec.last_touch = t;
    }
    const double age = static_cast<double>(t - rec.last_touch);
    double R = __dsub_rn(1.0, __ddiv_rn(age, static_cast<double>(sa.W)));
    R = fmin(fmax(R, 0.0), 1.0);
    const double N = (b == 0 || b + 1 == nb) ? 1.0 : 0.0;
    const double P = __dadd_rn(__dadd_rn(__dmul_rn(sa.wR, R), __dmul_rn(sa.wE, E)), __dmul_rn(sa.wN, N));
    rec.score = E;
    rec.prio = P;
    rec.tier = P >= sa.hi ? 0 : (P >= sa.lo ? 1 : 2);
    rec.mass = mass;
    *dst = rec;
}

__device__ __forceinline__ void score_record(const ScoreArgs &sa, kvs_record *recs, size_t idx, uint64_t seq_id,
                                             uint32_t b, uint32_t nb, uint64_t t, float mass, uint32_t *err)
{
    score_loaded(sa, recs[idx], recs + idx, seq_id, b, nb, t, mass, err);
}

}  // namespace kvs
