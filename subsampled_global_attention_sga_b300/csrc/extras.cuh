// extras.cuh -- the two SGA components beside the kept set S, for one query row.
//
// "AVGGT: Rethinking Global Attention for Accelerating VGGT", Key design 3: the attention of a
// query is split into three disjoint components normalised by one softmax -- the kept set S,
// the token's own key (diagonal) and one mean key/value standing for every dropped patch.
// "RegimeVGGT ...", Key design 2: a key standing for g tokens carries the logit bias ln g.
//
// Readings: the diagonal term exists only for a dropped query; under SGA_MEAN_LOO a dropped
// query's mean leaves its own token out (count c-1), a kept query's mean covers all c dropped
// tokens; SGA_MEAN_GLOBAL uses all c for every query.  No mean term when its count is 0.
// Logits here are in the base-2 domain: s2 = log2(e) * (scale * q.k + ln count).
#pragma once

#include "rope.cuh"

namespace sga {

struct ExtraArgs {
    int on;                 // 1: SGA with the extra components evaluated
    int diag, mean, mean_mode;
    long long dropped;      // c = |D| per (batch, head)
    long long T;            // tokens per (batch, head)
    const int32_t* slot;    // [T]: slot of a kept token in K_S, -1 if dropped
    const void* K;          // [BH, T, 64] full keys (dropped rows are read)
    const void* V;          // [BH, T, 64] full values
    const float* k_sum;     // [BH, 64] sums of the dropped keys
    const float* v_sum;     // [BH, 64] sums of the dropped values
    RopeArgs rope;          // rope.on: keys (and the caller's q) are rotated; k_sum already is
};

struct ExtraRow {
    float s_diag;   // base-2 logit of the diagonal term, -inf if absent
    float s_mean;   // base-2 logit of the mean term, -inf if absent
    int loo;        // 1: the mean leaves this row's own token out
    float inv_c;    // 1 / count of the mean term
};

// Logits of the extra components of query row i (token i of pair bh) with query q (already
// rotated when kRope); with kRope the key row k_i is rotated here (k_sum already is).
template <typename T, bool kRope = false>
__device__ __forceinline__ ExtraRow extra_logits(const ExtraArgs& a, int bh, long long i,
                                                 const float (&q)[64], float scale_log2) {
    ExtraRow r;
    r.s_diag = -INFINITY;
    r.s_mean = -INFINITY;
    r.loo = 0;
    r.inv_c = 0.f;
    if (!SGA_CHECK_INDEX(i, a.T, 11)) return r;
    const bool dropped_row = a.slot[i] < 0;
    const T* krow = reinterpret_cast<const T*>(a.K) + ((long long)bh * a.T + i) * 64;
    if (a.diag && dropped_row) {
        float kk[64];
        load_row64<T>(krow, kk);
        if (kRope) rope_row64(a.rope, i, kk);
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) s = fmaf(q[j], kk[j], s);
        r.s_diag = s * scale_log2;
    }
    if (a.mean) {
        const bool loo = (a.mean_mode == SGA_MEAN_LOO) && dropped_row;
        const long long ci = a.dropped - (loo ? 1 : 0);
        if (ci > 0) {
            const float* ks = a.k_sum + (long long)bh * 64;
            float kk[64];
            if (loo) {
                load_row64<T>(krow, kk);
                if (kRope) rope_row64(a.rope, i, kk);
            }
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const float kb = loo ? (__ldg(ks + j) - kk[j]) : __ldg(ks + j);
                s = fmaf(q[j], kb, s);
            }
            r.inv_c = 1.0f / (float)ci;
            r.loo = loo ? 1 : 0;
            // scale*q.kbar + ln(ci), to base 2: scale_log2 * q.kbar + log2(ci)
            r.s_mean = s * r.inv_c * scale_log2 + log2f((float)ci);
        }
    }
    return r;
}

// Add w_diag * v_i + w_mean * vbar_i to o[c0 .. c0+n) given the row's final base-2 max m.
template <typename T, int NCOL>
__device__ __forceinline__ void extra_values(const ExtraArgs& a, int bh, long long i,
                                             const ExtraRow& r, float m, int c0, float* o) {
    const T* vrow = reinterpret_cast<const T*>(a.V) + ((long long)bh * a.T + i) * 64;
    const float* vs = a.v_sum + (long long)bh * 64;
    const float wd = (r.s_diag == -INFINITY) ? 0.f : exp2f(r.s_diag - m);
    const float wm = (r.s_mean == -INFINITY) ? 0.f : exp2f(r.s_mean - m) * r.inv_c;
    if (wd == 0.f && wm == 0.f) return;
    const bool need_v = (wd != 0.f) || r.loo;
#pragma unroll
    for (int j = 0; j < NCOL; ++j) {
        const float vi = need_v ? Elem<T>::to_f(vrow[c0 + j]) : 0.f;
        const float vsum = __ldg(vs + c0 + j) - (r.loo ? vi : 0.f);
        o[j] = fmaf(wd, vi, fmaf(wm, vsum, o[j]));
    }
}

}  // namespace sga
