// compact.cuh -- the SGA compaction step: one streaming pass over K and V that copies the
// kept rows into contiguous K_S / V_S and sums the dropped rows.
//
// "AVGGT: Rethinking Global Attention for Accelerating VGGT", Key design 2: K and V are
// replaced by their subset S; Key design 3: one mean key/value stands for all dropped patches
// (the sums formed here; the division by the count happens in the attention kernel).
//
// HBM-bound.  Each 64-wide row is read with 16-byte vector loads by a group of lanes (8 lanes
// for bf16, 16 for fp32); several rows per lane are in flight.  Kept rows go to the slot the
// plan assigned; dropped rows are accumulated in fp32 registers.  The per-block partial sums go
// to a scratch buffer and a second kernel adds them in a fixed order, so the result does not
// depend on scheduling.
#pragma once

#include "rope.cuh"

namespace sga {

constexpr int kCompactThreads = 256;
constexpr int kCompactUnroll = 4;

struct CompactArgs {
    long long T;            // tokens per (batch, head)
    long long S;            // kept tokens per (batch, head)
    int rows_per_chunk;     // tokens handled by one block
    int n_chunks;           // blocks per (batch, head)
    const int32_t* slot;    // [T]
    const void* K;
    const void* V;
    void* KS;
    void* VS;
    float* partials;        // [BH, n_chunks, 128] (64 key sums, then 64 value sums)
    RopeArgs rope;          // with kRope: keys are rotated before they are stored or summed
};

// 16-byte vector of T <-> its E = 16 / sizeof(T) elements as fp32
template <typename T> struct Vec16;
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int E = 8;
    static __device__ __forceinline__ void unpack(const uint4& v, float (&x)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) { x[2 * i] = bf16_lo(w[i]); x[2 * i + 1] = bf16_hi(w[i]); }
    }
    static __device__ __forceinline__ uint4 pack(const float (&x)[8]) {
        return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                          pack_bf16x2(x[6], x[7]));
    }
};
template <> struct Vec16<float> {
    static constexpr int E = 4;
    static __device__ __forceinline__ void unpack(const uint4& v, float (&x)[4]) {
        x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
    }
    static __device__ __forceinline__ uint4 pack(const float (&x)[4]) {
        return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]));
    }
};

template <typename T, bool kRope>
__global__ void __launch_bounds__(kCompactThreads) compact_kernel(CompactArgs a) {
    constexpr int kLanesPerRow = 64 * (int)sizeof(T) / 16;     // 8 (bf16) or 16 (fp32)
    constexpr int kRowsPerPass = kCompactThreads / kLanesPerRow;
    constexpr int kElemsPerVec = 16 / (int)sizeof(T);            // 8 or 4
    __shared__ float red[kCompactThreads][2 * kElemsPerVec + 1];

    const int chunk = blockIdx.x;
    const int bh = blockIdx.y;
    const int vec = threadIdx.x % kLanesPerRow;
    const int rsub = threadIdx.x / kLanesPerRow;

    const uint4* K = reinterpret_cast<const uint4*>(a.K) + (long long)bh * a.T * kLanesPerRow;
    const uint4* V = reinterpret_cast<const uint4*>(a.V) + (long long)bh * a.T * kLanesPerRow;
    uint4* KS = reinterpret_cast<uint4*>(a.KS) + (long long)bh * a.S * kLanesPerRow;
    uint4* VS = reinterpret_cast<uint4*>(a.VS) + (long long)bh * a.S * kLanesPerRow;

    float ks[kElemsPerVec], vs[kElemsPerVec];
#pragma unroll
    for (int e = 0; e < kElemsPerVec; ++e) { ks[e] = 0.f; vs[e] = 0.f; }

    const long long r_begin = (long long)chunk * a.rows_per_chunk;
    const long long r_end = (r_begin + a.rows_per_chunk < a.T) ? r_begin + a.rows_per_chunk : a.T;

    if constexpr (kRope) {
        // rotated keys: the (cos, sin) table in shared memory; every lane takes part in each
        // row group's shuffles, rows past the chunk end with zeros
        extern __shared__ float2 rope_s[];
        for (int i = threadIdx.x; i < a.rope.P * 16; i += kCompactThreads) rope_s[i] = a.rope.tab[i];
        __syncthreads();
        using VT = Vec16<T>;
        for (long long r0 = r_begin; r0 < r_end; r0 += (long long)kRowsPerPass * kCompactUnroll) {
            uint4 kv[kCompactUnroll], vv[kCompactUnroll];
            int sl[kCompactUnroll];
#pragma unroll
            for (int u = 0; u < kCompactUnroll; ++u) {
                const long long t = r0 + (long long)u * kRowsPerPass + rsub;
                sl[u] = -2;
                kv[u] = make_uint4(0u, 0u, 0u, 0u);
                vv[u] = kv[u];
                if (t < r_end) {
                    sl[u] = __ldg(a.slot + t);
                    kv[u] = __ldcs(K + t * kLanesPerRow + vec);
                    vv[u] = __ldcs(V + t * kLanesPerRow + vec);
                }
            }
#pragma unroll
            for (int u = 0; u < kCompactUnroll; ++u) {
                const long long t = r0 + (long long)u * kRowsPerPass + rsub;
                int pr, pc;
                rope_pos(a.rope, t < r_end ? t : 0, pr, pc);
                float xk[kElemsPerVec], xv[kElemsPerVec];
                VT::unpack(kv[u], xk);
                rope_lane<kElemsPerVec>(rope_s, pr, pc, vec * kElemsPerVec, xk);
                if (sl[u] >= 0) {
                    KS[(long long)sl[u] * kLanesPerRow + vec] = VT::pack(xk);
                    VS[(long long)sl[u] * kLanesPerRow + vec] = vv[u];
                } else if (sl[u] == -1) {
                    VT::unpack(vv[u], xv);
#pragma unroll
                    for (int e = 0; e < kElemsPerVec; ++e) { ks[e] += xk[e]; vs[e] += xv[e]; }
                }
            }
        }
    } else {
    for (long long r0 = r_begin; r0 < r_end; r0 += (long long)kRowsPerPass * kCompactUnroll) {
        uint4 kv[kCompactUnroll], vv[kCompactUnroll];
        int sl[kCompactUnroll];
#pragma unroll
        for (int u = 0; u < kCompactUnroll; ++u) {
            const long long t = r0 + (long long)u * kRowsPerPass + rsub;
            sl[u] = -2;
            if (t < r_end) {
                sl[u] = __ldg(a.slot + t);
                kv[u] = __ldcs(K + t * kLanesPerRow + vec);
                vv[u] = __ldcs(V + t * kLanesPerRow + vec);
            }
        }
#pragma unroll
        for (int u = 0; u < kCompactUnroll; ++u) {
            if (sl[u] >= 0) {
                KS[(long long)sl[u] * kLanesPerRow + vec] = kv[u];
                VS[(long long)sl[u] * kLanesPerRow + vec] = vv[u];
            } else if (sl[u] == -1) {
                if constexpr (sizeof(T) == 2) {
                    const uint32_t kw[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
                    const uint32_t vw[4] = {vv[u].x, vv[u].y, vv[u].z, vv[u].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        ks[2 * e] += bf16_lo(kw[e]);
                        ks[2 * e + 1] += bf16_hi(kw[e]);
                        vs[2 * e] += bf16_lo(vw[e]);
                        vs[2 * e + 1] += bf16_hi(vw[e]);
                    }
                } else {
                    ks[0] += __uint_as_float(kv[u].x); ks[1] += __uint_as_float(kv[u].y);
                    ks[2] += __uint_as_float(kv[u].z); ks[3] += __uint_as_float(kv[u].w);
                    vs[0] += __uint_as_float(vv[u].x); vs[1] += __uint_as_float(vv[u].y);
                    vs[2] += __uint_as_float(vv[u].z); vs[3] += __uint_as_float(vv[u].w);
                }
            }
        }
    }
    }

#pragma unroll
    for (int e = 0; e < kElemsPerVec; ++e) {
        red[threadIdx.x][e] = ks[e];
        red[threadIdx.x][kElemsPerVec + e] = vs[e];
    }
    __syncthreads();
    // 128 outputs: dim j of the key sum (j < 64) or of the value sum (j >= 64); added over the
    // threads that hold that dim, in thread order.
    if (threadIdx.x < 128) {
        const int which = threadIdx.x >> 6;          // 0: keys, 1: values
        const int dim = threadIdx.x & 63;
        const int v = dim / kElemsPerVec, e = dim % kElemsPerVec;
        float s = 0.f;
        for (int r = 0; r < kRowsPerPass; ++r) s += red[r * kLanesPerRow + v][which * kElemsPerVec + e];
        a.partials[((long long)bh * a.n_chunks + chunk) * 128 + threadIdx.x] = s;
    }
}

// k_sum/v_sum[bh][d] = sum over chunks (in order) of the partials.
__global__ void __launch_bounds__(128) compact_finalize_kernel(const float* partials, int n_chunks,
                                                               float* k_sum, float* v_sum) {
    const int bh = blockIdx.x;
    const int j = threadIdx.x;
    const float* p = partials + (long long)bh * n_chunks * 128 + j;
    float s = 0.f;
    for (int c = 0; c < n_chunks; ++c) s += p[(long long)c * 128];
    if (j < 64) k_sum[bh * 64 + j] = s;
    else v_sum[bh * 64 + (j - 64)] = s;
}

}  // namespace sga
