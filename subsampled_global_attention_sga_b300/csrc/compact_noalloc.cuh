// compact_noalloc.cuh -- the compaction kernel of sga_compact_noalloc: the same streaming pass
// as compact_kernel (kept rows copied into K_S / V_S, dropped rows summed in fp32, per-block
// partial sums written to scratch), except that a token's slot in K_S is derived from the layer
// configuration in closed form instead of being read from a plan's slot map.  The caller then
// needs no plan, and so no device allocation at all.
//
// The kept set is the one of "AVGGT: Rethinking Global Attention for Accelerating VGGT", Key
// design 2 (the first patch of every s_h x s_w window, special tokens and -- for VGGT -- frame 0
// kept) with the per-frame phase shift of "RegimeVGGT ...", Key design 3: row offset
// (f div s_w) mod s_h, column offset f mod s_w.  Within a frame the kept tokens keep their
// order: the special tokens first, then the kept patches row by row.
#pragma once

#include "common.cuh"

namespace sga {

struct NoallocArgs {
    long long T;            // tokens per (batch, head)
    long long S;            // kept tokens per (batch, head)
    int L;                  // tokens per frame
    int n_special, grid_h, grid_w, s_h, s_w, phase_shift, ref_frame_dense;
    int rows_per_chunk;     // tokens handled by one block
    int n_chunks;           // blocks per (batch, head)
    const void* K;
    const void* V;
    void* KS;
    void* VS;
    float* partials;        // [BH, n_chunks, 128] (64 key sums, then 64 value sums)
};

__device__ __forceinline__ bool na_frame_dense(const NoallocArgs& a, int f) {
    return (f == 0 && a.ref_frame_dense) || (a.s_h == 1 && a.s_w == 1);
}

__device__ __forceinline__ void na_phase(const NoallocArgs& a, int f, int& pr, int& pc) {
    pr = a.phase_shift ? (f / a.s_w) % a.s_h : 0;
    pc = a.phase_shift ? f % a.s_w : 0;
}

// kept patch columns of a frame whose column phase is pc
__device__ __forceinline__ long long na_kept_cols(const NoallocArgs& a, int pc) {
    return pc < a.grid_w ? (a.grid_w - pc + a.s_w - 1) / a.s_w : 0;
}

__device__ __forceinline__ long long na_kept_in_frame(const NoallocArgs& a, int f) {
    if (na_frame_dense(a, f)) return a.L;
    int pr, pc;
    na_phase(a, f, pr, pc);
    const long long rows = pr < a.grid_h ? (a.grid_h - pr + a.s_h - 1) / a.s_h : 0;
    return a.n_special + rows * na_kept_cols(a, pc);
}

// Kept tokens of frames 0 .. f-1.  Frames 1, 2, ... repeat their phase every s_h*s_w frames
// (every frame without the phase shift), so they are counted per residue class.
__device__ long long na_frame_offset(const NoallocArgs& a, int f) {
    if (f <= 0) return 0;
    long long off = na_kept_in_frame(a, 0);
    const int period = a.phase_shift ? a.s_h * a.s_w : 1;
    for (int r = 0; r < period; ++r) {
        const int first = (r == 0) ? period : r;      // smallest frame >= 1 with this residue
        if (first > f - 1) continue;
        const long long n = (long long)(f - 1 - first) / period + 1;
        off += n * na_kept_in_frame(a, first);
    }
    return off;
}

// Slot of token t in K_S, or -1 if t is dropped.  (cf, coff) cache the last frame's offset.
__device__ __forceinline__ long long na_slot(const NoallocArgs& a, long long t, int& cf, long long& coff) {
    const int f = (int)(t / a.L);
    const int p = (int)(t - (long long)f * a.L);
    if (f != cf) {
        cf = f;
        coff = na_frame_offset(a, f);
    }
    if (na_frame_dense(a, f) || p < a.n_special) return coff + p;
    const int q = p - a.n_special;
    const int r = q / a.grid_w, c = q - r * a.grid_w;
    int pr, pc;
    na_phase(a, f, pr, pc);
    if (r < pr || c < pc || (r - pr) % a.s_h != 0 || (c - pc) % a.s_w != 0) return -1;
    return coff + a.n_special + (long long)((r - pr) / a.s_h) * na_kept_cols(a, pc) + (c - pc) / a.s_w;
}

template <typename T>
__global__ void __launch_bounds__(kCompactThreads) compact_noalloc_kernel(NoallocArgs a) {
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
    int cf = -1;
    long long coff = 0;

    for (long long r0 = r_begin; r0 < r_end; r0 += (long long)kRowsPerPass * kCompactUnroll) {
        uint4 kv[kCompactUnroll], vv[kCompactUnroll];
        long long sl[kCompactUnroll];
#pragma unroll
        for (int u = 0; u < kCompactUnroll; ++u) {
            const long long t = r0 + (long long)u * kRowsPerPass + rsub;
            sl[u] = -2;
            if (t < r_end) {
                sl[u] = na_slot(a, t, cf, coff);
                kv[u] = __ldcs(K + t * kLanesPerRow + vec);
                vv[u] = __ldcs(V + t * kLanesPerRow + vec);
            }
        }
#pragma unroll
        for (int u = 0; u < kCompactUnroll; ++u) {
            if (sl[u] >= 0) {
                if (SGA_CHECK_INDEX(sl[u], a.S, 2) && sl[u] < a.S) {   // true for a consistent configuration
                    KS[sl[u] * kLanesPerRow + vec] = kv[u];
                    VS[sl[u] * kLanesPerRow + vec] = vv[u];
                }
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

#pragma unroll
    for (int e = 0; e < kElemsPerVec; ++e) {
        red[threadIdx.x][e] = ks[e];
        red[threadIdx.x][kElemsPerVec + e] = vs[e];
    }
    __syncthreads();
    // every block writes all 128 of its partials, so the scratch needs no clearing
    if (threadIdx.x < 128) {
        const int which = threadIdx.x >> 6;
        const int dim = threadIdx.x & 63;
        const int v = dim / kElemsPerVec, e = dim % kElemsPerVec;
        float s = 0.f;
        for (int r = 0; r < kRowsPerPass; ++r) s += red[r * kLanesPerRow + v][which * kElemsPerVec + e];
        a.partials[((long long)bh * a.n_chunks + chunk) * 128 + threadIdx.x] = s;
    }
}

}  // namespace sga
