// attn_simt.cuh -- CUDA-core attention kernel (fp32 arithmetic) for every variant: SGA over
// the compacted keys plus the diagonal/mean components, dense global attention, and
// frame-local attention.  It is the fp32 path (fp32 I/O, accurate exp2f) and the independent
// CUDA-core cross-check of the tensor-core kernel for bf16 I/O.
//
// One thread owns one query row: q and the output accumulator live in registers; keys and
// values are staged 64 at a time in shared memory (as fp32) and read by broadcast.  The
// softmax is the standard online form ("AVGGT ..." Key design 2, softmax(QK^T/sqrt(d))V) in
// the base-2 domain.
#pragma once

#include "extras.cuh"

namespace sga {

struct SimtArgs {
    long long seg_rows;       // query rows per segment
    long long kv_rows;        // keys per segment
    const void* Q;            // [n_seg, seg_rows, 64]
    const void* Kt;           // [n_seg, kv_rows, 64] keys attended (K_S, K, or frames of K)
    const void* Vt;
    void* O;                  // [n_seg, seg_rows, 64]
    float* lse;               // [n_seg, seg_rows] or null
    float scale_log2;         // scale * log2(e)
    ExtraArgs ex;             // ex.on only for SGA (segment = batch*head)
    const float* bias;        // [n_seg, kv_rows] natural-log per-key bias, or null
};

constexpr int kSimtRows = 128;   // query rows (threads) per block
constexpr int kSimtKeys = 64;    // keys staged per round
constexpr int kSimtChunk = 16;   // keys per online-softmax update

template <typename T>
__global__ void __launch_bounds__(kSimtRows) attn_simt_kernel(SimtArgs p) {
    __shared__ float Ks[kSimtKeys][64];
    __shared__ float Vs[kSimtKeys][64];
    __shared__ float Bs[kSimtKeys];             // per-key bias in base 2 (0 without a bias)

    const int seg = blockIdx.y;
    const long long row = (long long)blockIdx.x * kSimtRows + threadIdx.x;
    const bool valid = row < p.seg_rows;

    const T* Qb = reinterpret_cast<const T*>(p.Q) + (long long)seg * p.seg_rows * 64;
    const T* Kb = reinterpret_cast<const T*>(p.Kt) + (long long)seg * p.kv_rows * 64;
    const T* Vb = reinterpret_cast<const T*>(p.Vt) + (long long)seg * p.kv_rows * 64;

    float q[64];
    if (valid) {
        load_row64<T>(Qb + row * 64, q);
        if (p.ex.rope.on) rope_row64(p.ex.rope, row, q);
    } else {
#pragma unroll
        for (int j = 0; j < 64; ++j) q[j] = 0.f;
    }

    float o[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) o[j] = 0.f;
    float m = -INFINITY, l = 0.f;

    ExtraRow xr{};
    if (p.ex.on && valid) {
        xr = p.ex.rope.on ? extra_logits<T, true>(p.ex, seg, row, q, p.scale_log2)
                          : extra_logits<T, false>(p.ex, seg, row, q, p.scale_log2);
        m = fmaxf(xr.s_diag, xr.s_mean);
        if (m != -INFINITY) {
            l = (xr.s_diag == -INFINITY ? 0.f : exp2f(xr.s_diag - m)) +
                (xr.s_mean == -INFINITY ? 0.f : exp2f(xr.s_mean - m));
        }
    }

    for (long long k0 = 0; k0 < p.kv_rows; k0 += kSimtKeys) {
        const long long rem = p.kv_rows - k0;
        const int nk = rem < kSimtKeys ? (int)rem : kSimtKeys;
        __syncthreads();
        for (int e = threadIdx.x; e < kSimtKeys * 64; e += kSimtRows) {
            const int r = e >> 6, c = e & 63;
            float kv = 0.f, vv = 0.f;
            if (r < nk) {
                kv = Elem<T>::to_f(Kb[(k0 + r) * 64 + c]);
                vv = Elem<T>::to_f(Vb[(k0 + r) * 64 + c]);
            }
            Ks[r][c] = kv;
            Vs[r][c] = vv;
        }
        if (threadIdx.x < kSimtKeys) {
            const int r = threadIdx.x;
            Bs[r] = (p.bias && r < nk) ? p.bias[(long long)seg * p.kv_rows + k0 + r] * 1.4426950408889634f : 0.f;
        }
        __syncthreads();
        for (int c0 = 0; c0 < nk; c0 += kSimtChunk) {
            float s[kSimtChunk];
            float mx = -INFINITY;
#pragma unroll
            for (int jj = 0; jj < kSimtChunk; ++jj) {
                float acc = 0.f;
#pragma unroll
                for (int d = 0; d < 64; ++d) acc = fmaf(q[d], Ks[c0 + jj][d], acc);
                s[jj] = (c0 + jj < nk) ? fmaf(acc, p.scale_log2, Bs[c0 + jj]) : -INFINITY;
                mx = fmaxf(mx, s[jj]);
            }
            const float m_new = fmaxf(m, mx);
            const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
            l *= alpha;
#pragma unroll
            for (int d = 0; d < 64; ++d) o[d] *= alpha;
#pragma unroll
            for (int jj = 0; jj < kSimtChunk; ++jj) {
                const float pj = exp2f(s[jj] - m_new);
                l += pj;
#pragma unroll
                for (int d = 0; d < 64; ++d) o[d] = fmaf(pj, Vs[c0 + jj][d], o[d]);
            }
            m = m_new;
        }
    }

    if (!valid) return;
    if (!SGA_CHECK_INDEX((long long)seg * p.seg_rows + row, (long long)gridDim.y * p.seg_rows, 12)) return;
    if (p.ex.on) extra_values<T, 64>(p.ex, seg, row, xr, m, 0, o);
    const float inv_l = 1.0f / l;
    T* Ob = reinterpret_cast<T*>(p.O) + ((long long)seg * p.seg_rows + row) * 64;
#pragma unroll
    for (int d = 0; d < 64; ++d) Ob[d] = Elem<T>::from_f(o[d] * inv_l);
    if (p.lse) p.lse[(long long)seg * p.seg_rows + row] = (m + log2f(l)) * 0.69314718055994531f;
}

}  // namespace sga
