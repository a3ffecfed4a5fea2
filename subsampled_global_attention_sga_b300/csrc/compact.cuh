// compact.cuh -- the SGA compaction step: one streaming pass over K and V that copies the
// kept rows into contiguous K_S / V_S and sums the dropped rows.
//
// "AVGGT: Rethinking Global Attention for Accelerating VGGT", Key design 2: K and V are
// replaced by their subset S; Key design 3: one mean key/value stands for all dropped patches
// (the sums formed here; the division by the count happens in the attention kernel).
//
// HBM-bound.  Each 64-wide row is read with 16-byte vector loads by a group of lanes (8 lanes
// for bf16, 16 for fp32; half as many with the rotation, each lane then holding the two vectors
// whose dims rotate together); several rows per lane are in flight.  Kept rows go to the slot the
// plan assigned; dropped rows are accumulated in fp32 registers.  The per-block partial sums go
// to a scratch buffer and a second kernel adds them in a fixed order, so the result does not
// depend on scheduling.  (bf16 with the rotation runs the TMA-fed kernel of compact_rope.cuh;
// this kernel's rotating instance serves fp32.)
#pragma once

#include "rope.cuh"

namespace sga {

constexpr int kCompactThreads = 256;
// (cos, sin) table rows in shared memory padded from 16 to 18 entries (144 bytes): the rows of
// the 8 tokens a warp rotates at once start 4 banks apart, and a row stays 16-byte aligned
constexpr int kRopeTabStride = 18;
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
__global__ void __launch_bounds__(kCompactThreads, kRope ? 2 : 1) compact_kernel(CompactArgs a) {
    constexpr int kLanesPerRow = 64 * (int)sizeof(T) / 16;     // 16-byte vectors per row: 8 (bf16) or 16 (fp32)
    constexpr int kElemsPerVec = 16 / (int)sizeof(T);            // 8 or 4
    // with the rotation a lane holds both vectors of its rotation pairs (dims j and j+16 of a
    // 32-dim half), so a row takes half as many lanes and no shuffles
    constexpr int kRowLanes = kRope ? kLanesPerRow / 2 : kLanesPerRow;
    constexpr int kVecsPerLane = kRope ? 2 : 1;
    constexpr int kRowsPerPass = kCompactThreads / kRowLanes;
    constexpr int kSums = kVecsPerLane * kElemsPerVec;            // key (and value) sums per lane
    // rows in flight per lane (a rotating lane moves two vectors of K and of V per row; three
    // rows keep it within two blocks per SM)
    constexpr int kUnroll = kRope ? 3 : kCompactUnroll;
    __shared__ float red[kCompactThreads][2 * kSums + 1];

    const int chunk = blockIdx.x;
    const int bh = blockIdx.y;
    const int lane_r = threadIdx.x % kRowLanes;
    const int rsub = threadIdx.x / kRowLanes;
    // vectors of this lane: without the rotation one (lane_r); with it the pair (va, va + PO),
    // PO = 16 dims in vectors, va running over the first 16 dims of each 32-dim half
    constexpr int PO = 16 / kElemsPerVec;
    const int va = kRope ? (lane_r % PO) + 2 * PO * (lane_r / PO) : lane_r;

    const uint4* K = reinterpret_cast<const uint4*>(a.K) + (long long)bh * a.T * kLanesPerRow;
    const uint4* V = reinterpret_cast<const uint4*>(a.V) + (long long)bh * a.T * kLanesPerRow;
    uint4* KS = reinterpret_cast<uint4*>(a.KS) + (long long)bh * a.S * kLanesPerRow;
    uint4* VS = reinterpret_cast<uint4*>(a.VS) + (long long)bh * a.S * kLanesPerRow;

    float ks[kSums], vs[kSums];
#pragma unroll
    for (int e = 0; e < kSums; ++e) { ks[e] = 0.f; vs[e] = 0.f; }

    const long long r_begin = (long long)chunk * a.rows_per_chunk;
    const long long r_end = (r_begin + a.rows_per_chunk < a.T) ? r_begin + a.rows_per_chunk : a.T;

    if constexpr (kRope) {
        // rotated keys: the (cos, sin) table in shared memory
        extern __shared__ float2 rope_s[];
        for (int i = threadIdx.x; i < a.rope.P * 16; i += kCompactThreads)
            rope_s[(i >> 4) * kRopeTabStride + (i & 15)] = a.rope.tab[i];
        __syncthreads();
        using VT = Vec16<T>;
        const int d0 = va * kElemsPerVec;                         // first dim of vector va
        // token position within its frame, per row in flight, stepped along with the rows (no
        // division per row); the grid row of a patch from a float quotient that is exact for the
        // frame sizes the plan allows (q < 2^21)
        constexpr int kStep = kRowsPerPass * kUnroll;
        const int L = a.rope.L, ns = a.rope.n_special, gw = a.rope.grid_w, off = a.rope.pos_offset;
        const int step_mod = kStep % L;
        const float inv_gw = 1.0f / (float)gw;
        int pu[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) pu[u] = (int)((r_begin + (long long)u * kRowsPerPass + rsub) % L);
        for (long long r0 = r_begin; r0 < r_end; r0 += (long long)kRowsPerPass * kUnroll) {
            uint4 ka[kUnroll], kb[kUnroll], wa[kUnroll], wb[kUnroll];
            int sl[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const long long t = r0 + (long long)u * kRowsPerPass + rsub;
                sl[u] = -2;
                if (t < r_end) {
                    sl[u] = __ldg(a.slot + t);
                    ka[u] = __ldcs(K + t * kLanesPerRow + va);
                    kb[u] = __ldcs(K + t * kLanesPerRow + va + PO);
                    wa[u] = __ldcs(V + t * kLanesPerRow + va);
                    wb[u] = __ldcs(V + t * kLanesPerRow + va + PO);
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (sl[u] == -2) continue;
                int pr = 0, pc = 0;
                if (pu[u] >= ns) {
                    const int q = pu[u] - ns;
                    const int qr = (int)(((float)q + 0.5f) * inv_gw);
                    pr = qr + off;
                    pc = q - qr * gw + off;
                }
                const float2* tb = rope_s + ((d0 & 32) ? pc : pr) * kRopeTabStride + (d0 & 15);
                float x0[kElemsPerVec], x1[kElemsPerVec];
                VT::unpack(ka[u], x0);
                VT::unpack(kb[u], x1);
#pragma unroll
                for (int e = 0; e < kElemsPerVec; ++e) {             // dims d0+e and d0+e+16
                    const float2 cs = tb[e];
                    const float y0 = fmaf(-x1[e], cs.y, x0[e] * cs.x);
                    const float y1 = fmaf(x0[e], cs.y, x1[e] * cs.x);
                    x0[e] = y0;
                    x1[e] = y1;
                }
                if (sl[u] >= 0) {
                    if (!SGA_CHECK_INDEX(sl[u], a.S, 1)) continue;
                    uint4* ksr = KS + (long long)sl[u] * kLanesPerRow;
                    uint4* vsr = VS + (long long)sl[u] * kLanesPerRow;
                    ksr[va] = VT::pack(x0);
                    ksr[va + PO] = VT::pack(x1);
                    vsr[va] = wa[u];
                    vsr[va + PO] = wb[u];
                } else {
                    float v0[kElemsPerVec], v1[kElemsPerVec];
                    VT::unpack(wa[u], v0);
                    VT::unpack(wb[u], v1);
#pragma unroll
                    for (int e = 0; e < kElemsPerVec; ++e) {
                        ks[e] += x0[e];
                        ks[kElemsPerVec + e] += x1[e];
                        vs[e] += v0[e];
                        vs[kElemsPerVec + e] += v1[e];
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                pu[u] += step_mod;
                if (pu[u] >= L) pu[u] -= L;
            }
        }
    } else {
    for (long long r0 = r_begin; r0 < r_end; r0 += (long long)kRowsPerPass * kUnroll) {
        uint4 kv[kUnroll], vv[kUnroll];
        int sl[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long t = r0 + (long long)u * kRowsPerPass + rsub;
            sl[u] = -2;
            if (t < r_end) {
                sl[u] = __ldg(a.slot + t);
                kv[u] = __ldcs(K + t * kLanesPerRow + va);
                vv[u] = __ldcs(V + t * kLanesPerRow + va);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (sl[u] >= 0) {
                if (!SGA_CHECK_INDEX(sl[u], a.S, 1)) continue;
                KS[(long long)sl[u] * kLanesPerRow + va] = kv[u];
                VS[(long long)sl[u] * kLanesPerRow + va] = vv[u];
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
    for (int e = 0; e < kSums; ++e) {
        red[threadIdx.x][e] = ks[e];
        red[threadIdx.x][kSums + e] = vs[e];
    }
    __syncthreads();
    // 128 outputs: dim j of the key sum (j < 64) or of the value sum (j >= 64); added over the
    // threads that hold that dim, in thread order.
    if (threadIdx.x < 128) {
        const int which = threadIdx.x >> 6;          // 0: keys, 1: values
        const int dim = threadIdx.x & 63;
        const int v = dim / kElemsPerVec, e = dim % kElemsPerVec;
        // the lane holding vector v, and which of its vectors it is
        int lane_v = v, slot_v = 0;
        if (kRope) {
            const int h = v / (2 * PO), w = v % (2 * PO);
            slot_v = w / PO;
            lane_v = (w % PO) + PO * h;
        }
        float s = 0.f;
        for (int r = 0; r < kRowsPerPass; ++r)
            s += red[r * kRowLanes + lane_v][which * kSums + slot_v * kElemsPerVec + e];
        a.partials[((long long)bh * a.n_chunks + chunk) * 128 + threadIdx.x] = s;
    }
}

// k_sum/v_sum[bh][d] = the partials in a fixed order: the chunks cut into kFinalizeRuns
// consecutive runs, each summed in chunk order by its own thread, then the run sums in order.
// (One chain over all the chunks made the sum a long series of dependent loads.)
constexpr int kFinalizeRuns = 8;
__global__ void __launch_bounds__(128 * kFinalizeRuns) compact_finalize_kernel(const float* partials, int n_chunks,
                                                                               float* k_sum, float* v_sum) {
    __shared__ float run_sum[kFinalizeRuns][128];
    const int bh = blockIdx.x;
    const int j = threadIdx.x & 127, run = threadIdx.x >> 7;
    const int c0 = (int)((long long)run * n_chunks / kFinalizeRuns);
    const int c1 = (int)((long long)(run + 1) * n_chunks / kFinalizeRuns);
    const float* p = partials + (long long)bh * n_chunks * 128 + j;
    float s = 0.f;
    for (int c = c0; c < c1; ++c) s += p[(long long)c * 128];
    run_sum[run][j] = s;
    __syncthreads();
    if (threadIdx.x < 128) {
        float t = 0.f;
        for (int r = 0; r < kFinalizeRuns; ++r) t += run_sum[r][j];
        if (j < 64) k_sum[bh * 64 + j] = t;
        else v_sum[bh * 64 + (j - 64)] = t;
    }
}

}  // namespace sga
