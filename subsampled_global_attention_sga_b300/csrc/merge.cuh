// merge.cuh -- head-wise temporal token merging and unmerging (d = 64).
//
// "HTTM: Head-wise Temporal Token Merging for Faster VGGT" (blog digest), section 2: each head
// merges its own tokens; tokens are grouped into temporal blocks (the same spatial run of
// patches over consecutive frames) and merged inside a block only; the first frame anchors
// (its tokens are the destinations); values follow the keys' matching; unmerging copies a
// merged token's output back to every token it stands for.  "RegimeVGGT ..." Key design 2: a
// merged token standing for g tokens carries the logit bias ln g (size-aware attention).
//
// Reading (identical in the test oracle): frames in chunks of n_t; a block = the run of n_s
// consecutive patch tokens [w*n_s, (w+1)*n_s) of every frame of one chunk; destinations = the
// chunk's first frame, sources = its other frames; special tokens are never merged.  Each
// source joins the destination with the largest cosine (first maximum), the
// r = floor(#sources * r_permille / 1000) most similar sources of the block are merged (ties:
// lower token index).  The cosine is decided in IEEE fp32 with one fixed order: norm =
// sqrt_rn(fma chain of x_i^2), dot = fma chain, cos = dot / (n_a * n_b) (0 if that is 0).
//
// Merged sequence (per (batch, head)), block-major: for each chunk, its special tokens (token
// order), then for each window its kept tokens (destinations and unmerged sources, token order).
// Every block's offset is a closed form, so no scan is needed.
#pragma once

#include "common.cuh"

namespace sga {

struct MergeGeom {
    int N, L, P, n_special, n_t, n_s, r_permille;
    int n_chunks, n_windows;
    long long T, M;
};

__host__ __device__ inline long long merge_kept_window(int nf, int ws, int r_permille) {
    return (long long)nf * ws - ((long long)(nf - 1) * ws * r_permille) / 1000;
}
__host__ __device__ inline int merge_window_size(const MergeGeom& g, int w) {
    return (w + 1) * g.n_s <= g.P ? g.n_s : g.P - w * g.n_s;
}
__host__ __device__ inline long long merge_chunk_size(const MergeGeom& g, int nf) {
    const int last = g.n_windows - 1;
    return (long long)nf * g.n_special + (long long)last * merge_kept_window(nf, g.n_s, g.r_permille) +
           merge_kept_window(nf, merge_window_size(g, last), g.r_permille);
}
// first merged index of window w (w = -1: the chunk's special tokens) of chunk c
__host__ __device__ inline long long merge_block_base(const MergeGeom& g, int c, int w) {
    const int nf = (c + 1) * g.n_t <= g.N ? g.n_t : g.N - c * g.n_t;
    long long b = (long long)c * merge_chunk_size(g, g.n_t);
    if (w >= 0) b += (long long)nf * g.n_special + (long long)w * merge_kept_window(nf, g.n_s, g.r_permille);
    return b;
}

constexpr int kMergeThreads = 256;
constexpr int kMergeMaxBlock = 512;    // n_t * n_s

struct MergeArgs {
    MergeGeom g;
    const void* X;          // [BH, T, 64]  the keys (matched)
    const void* Y;          // [BH, T, 64]  values following the match, or null
    void* Xm;               // [BH, M, 64]
    void* Ym;               // [BH, M, 64] or null
    float* log_g;           // [BH, M] natural log of the group size, or null
    int32_t* map;           // [BH, T] merged index of every token
};

// grid: (n_windows + 1, n_chunks, BH); blockIdx.x == n_windows handles the chunk's specials.
// Dynamic shared memory: the block's rows as fp32 with a padded stride of 65 (conflict-free
// per-thread rows), then norms, similarities, destinations and ranks; sized for nb_max entries.
__host__ __device__ constexpr int merge_smem_bytes(int nb_max) { return nb_max * 65 * 4 + 4 * nb_max * 4; }

template <typename T>
__global__ void __launch_bounds__(kMergeThreads, 3) merge_kernel(MergeArgs a, int nb_max) {
    const MergeGeom& g = a.g;
    const int c = blockIdx.y;
    const long long bh = blockIdx.z;
    const int f0 = c * g.n_t;
    const int nf = (c + 1) * g.n_t <= g.N ? g.n_t : g.N - f0;
    const T* X = reinterpret_cast<const T*>(a.X) + bh * g.T * 64;
    const T* Y = a.Y ? reinterpret_cast<const T*>(a.Y) + bh * g.T * 64 : nullptr;
    T* Xm = reinterpret_cast<T*>(a.Xm) + bh * g.M * 64;
    T* Ym = a.Ym ? reinterpret_cast<T*>(a.Ym) + bh * g.M * 64 : nullptr;
    float* lg = a.log_g ? a.log_g + bh * g.M : nullptr;
    int32_t* map = a.map + bh * g.T;

    if ((int)blockIdx.x == g.n_windows) {
        // special tokens of the chunk's frames: copied, group size 1
        const long long base = merge_block_base(g, c, -1);
        for (int i = threadIdx.x; i < nf * g.n_special * 64; i += kMergeThreads) {
            const int k = i / 64, e = i % 64;
            const long long t = (long long)(f0 + k / g.n_special) * g.L + k % g.n_special;
            Xm[(base + k) * 64 + e] = X[t * 64 + e];
            if (Ym) Ym[(base + k) * 64 + e] = Y[t * 64 + e];
            if (e == 0) {
                map[t] = (int32_t)(base + k);
                if (lg) lg[base + k] = 0.f;
            }
        }
        return;
    }

    const int w = blockIdx.x;
    const int ws = merge_window_size(g, w);
    const int nb = nf * ws;                         // tokens of the block: frame-major, then patch
    const int n_src = (nf - 1) * ws;
    const long long r = ((long long)n_src * g.r_permille) / 1000;
    const long long base = merge_block_base(g, c, w);

    extern __shared__ uint8_t smem[];
    float* xs = reinterpret_cast<float*>(smem);                  // [nb][65] (padded rows)
    float* nrm = xs + nb_max * 65;                               // [nb]
    float* sim = nrm + nb_max;                                   // [n_src]
    int* best = reinterpret_cast<int*>(sim + nb_max);            // [n_src] block index of the destination
    int* rank = best + nb_max;                                   // [nb]: merged index within block, or -1

    auto tok = [&](int i) -> long long {                        // token of block entry i
        return (long long)(f0 + i / ws) * g.L + g.n_special + (long long)w * g.n_s + i % ws;
    };
    for (int i = threadIdx.x; i < nb * 64; i += kMergeThreads) {
        const int k = i / 64, e = i % 64;
        xs[k * 65 + e] = Elem<T>::to_f(X[tok(k) * 64 + e]);
    }
    __syncthreads();
    for (int k = threadIdx.x; k < nb; k += kMergeThreads) {
        float s = 0.f;
        for (int e = 0; e < 64; ++e) s = __fmaf_rn(xs[k * 65 + e], xs[k * 65 + e], s);
        nrm[k] = __fsqrt_rn(s);
    }
    __syncthreads();
    // every source (entries ws .. nb-1) finds its destination (entries 0 .. ws-1)
    for (int a2 = threadIdx.x; a2 < n_src; a2 += kMergeThreads) {
        const int k = ws + a2;
        float xk[64];                                            // the source row, in registers
#pragma unroll
        for (int e = 0; e < 64; ++e) xk[e] = xs[k * 65 + e];
        float bs = -INFINITY;
        int bd = -1;
        for (int d = 0; d < ws; ++d) {
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < 64; ++e) dot = __fmaf_rn(xk[e], xs[d * 65 + e], dot);
            const float den = __fmul_rn(nrm[k], nrm[d]);
            const float cs = den == 0.f ? 0.f : __fdiv_rn(dot, den);
            if (cs > bs) { bs = cs; bd = d; }
        }
        sim[a2] = bs;
        best[a2] = bd;
    }
    __syncthreads();
    // merged sources: the r largest similarities (ties: lower token index = lower entry index,
    // since entries are in token order); kept entries get consecutive merged indices in token order
    for (int k = threadIdx.x; k < nb; k += kMergeThreads) {
        bool merged = false;
        if (k >= ws) {
            const int a2 = k - ws;
            long long ahead = 0;
            for (int b2 = 0; b2 < n_src; ++b2)
                if (sim[b2] > sim[a2] || (sim[b2] == sim[a2] && b2 < a2)) ++ahead;
            merged = ahead < r;
        }
        rank[k] = merged ? -1 : 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {                                     // kept entries in token order
        int m = 0;
        for (int k = 0; k < nb; ++k)
            if (rank[k] >= 0) rank[k] = m++;
    }
    __syncthreads();
    // group means: a kept entry plus the sources merged into it (destinations only), summed in
    // entry order, 16 dims at a time
    for (int k = threadIdx.x; k < nb; k += kMergeThreads) {
        const long long t = tok(k);
        if (rank[k] < 0) {
            map[t] = (int32_t)(base + rank[best[k - ws]]);
            continue;
        }
        const long long mi = base + rank[k];
        map[t] = (int32_t)mi;
        int cnt = 1;
        if (k < ws)
            for (int a2 = 0; a2 < n_src; ++a2) cnt += (rank[ws + a2] < 0 && best[a2] == k) ? 1 : 0;
        const float inv = 1.0f / (float)cnt;
        for (int e0 = 0; e0 < 64; e0 += 16) {
            float sx[16], sy[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                sx[e] = xs[k * 65 + e0 + e];
                sy[e] = Y ? Elem<T>::to_f(Y[t * 64 + e0 + e]) : 0.f;
            }
            if (k < ws && cnt > 1) {
                for (int a2 = 0; a2 < n_src; ++a2) {
                    if (rank[ws + a2] >= 0 || best[a2] != k) continue;
                    const long long ts = tok(ws + a2);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        sx[e] += xs[(ws + a2) * 65 + e0 + e];
                        if (Y) sy[e] += Elem<T>::to_f(Y[ts * 64 + e0 + e]);
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                Xm[mi * 64 + e0 + e] = Elem<T>::from_f(sx[e] * inv);
                if (Ym) Ym[mi * 64 + e0 + e] = Elem<T>::from_f(sy[e] * inv);
            }
        }
        if (lg) lg[mi] = logf((float)cnt);
    }
}


// Y[bh, t] = Ym[bh, map[bh, t]]: one thread per 16 bytes of a row.
template <typename T>
__global__ void __launch_bounds__(256) unmerge_kernel(const int32_t* map, const void* Ym, void* Y, long long T_seq,
                                                      long long M, long long rows_total) {
    constexpr int kVec = 64 * (int)sizeof(T) / 16;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows_total * kVec) return;
    const long long row = i / kVec;
    const int v = (int)(i % kVec);
    const long long bh = row / T_seq;
    const long long src = bh * M + __ldg(map + row);
    reinterpret_cast<uint4*>(Y)[row * kVec + v] = __ldg(reinterpret_cast<const uint4*>(Ym) + src * kVec + v);
}

}  // namespace sga
