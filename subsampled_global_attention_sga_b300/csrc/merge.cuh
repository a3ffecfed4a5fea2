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
    int nb_max;             // entries of the largest block (n_t * n_s)
    int y_smem;             // 1: the block's Y rows are staged in shared memory
};

// Dynamic shared memory of one block, sized for nb_max entries:
//   Y rows as stored (only when staged), X rows as fp32 with a padded stride of 68 floats (rows
//   16-byte aligned: a warp's per-thread float4 row reads are conflict-free and a destination
//   row is broadcast four values per load), norms, similarity / destination partials (at least
//   one per thread), and one bit per source that says whether it is merged.
constexpr int kXS = 68;                // row stride of the fp32 X rows in shared memory
__host__ __device__ constexpr int merge_partials(int nb_max) { return nb_max > kMergeThreads ? nb_max : kMergeThreads; }
__host__ __device__ constexpr int merge_smem_bytes(int nb_max, int elem_bytes, bool y_smem, bool x_f32 = true) {
    return (y_smem ? nb_max * 64 * elem_bytes : 0) +
           4 * ((x_f32 ? nb_max * kXS : 0) + nb_max + 2 * merge_partials(nb_max) + (nb_max + 31) / 32);
}

// The tensor-core matching (bf16 keys, at most 128 sources and 128 destinations per block): one
// tcgen05.mma computes every (source, destination) dot product at once, A = the block's source
// rows (128 x 64), B = its destination rows (Npad x 64), both in shared memory with the
// 128-byte swizzle, D in Tensor Memory.  Its fp32 sums come in the tensor core's order, so
// they only shortlist: a destination whose approximate cosine is within kMatchWindow of the
// best one gets the exact fixed-order fma chain, and the first maximum of the exact cosines
// decides, as before.  The window: the products of bf16 values are exact; an fp32 sum of 64 of
// them in any order is within 64 ulp-steps, under 2^-17 of sum |x_i b_i|, which Cauchy-Schwarz
// bounds by the product of the norms; so the approximate and exact cosines differ by less than
// 2^-16 (plus the divisions' rounding), and every destination whose exact cosine could reach
// the maximum lies within 2^-15 of the best approximate one.  kMatchWindow = 2^-10 leaves a
// factor 32 for the tensor core's accumulation order and rounding.
constexpr float kMatchWindow = 9.765625e-4f;          // 2^-10
constexpr int kTcMaxSrc = 128;                          // sources per block (one M = 128 tile)
constexpr int kTcMaxDst = 128;                          // destinations per block (N <= 128)
constexpr int kTcList = 8;                              // shortlist entries kept per source
__host__ __device__ constexpr int merge_tc_npad(int ws_max) { return ((ws_max + 15) / 16) * 16; }
// shared memory added by the tensor-core path: the A and B tiles (1024-byte aligned), the
// mbarrier and the TMEM address, the destinations' inverse norms and the sources' shortlists
__host__ __device__ constexpr int merge_tc_extra_bytes(int ws_max) {
    return 2048 + kTcMaxSrc * 128 + merge_tc_npad(ws_max) * 128 +   // + alignment slack
           4 * kTcMaxDst + kTcList * kTcMaxSrc;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// fp32 arithmetic on a bf16 operand taken straight from its half of a packed word: the
// mixed-precision fma / add of sm_100 and later round once, as fmaf / fadd of the operand
// widened to fp32 do (the widening is exact), so the results are the same bits
__device__ __forceinline__ float fma_bf16_lo(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %3;}" : "=f"(d) : "r"(a), "r"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fma_bf16_hi(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %3;}" : "=f"(d) : "r"(a), "r"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float add_bf16_lo(uint32_t a, float c) {
    float d;
    asm("{.reg .b16 al, ah;\n\tmov.b32 {al, ah}, %1;\n\tadd.rn.f32.bf16 %0, al, %2;}" : "=f"(d) : "r"(a), "f"(c));
    return d;
}
__device__ __forceinline__ float add_bf16_hi(uint32_t a, float c) {
    float d;
    asm("{.reg .b16 al, ah;\n\tmov.b32 {al, ah}, %1;\n\tadd.rn.f32.bf16 %0, ah, %2;}" : "=f"(d) : "r"(a), "f"(c));
    return d;
}
// the dot product of two 8-element bf16 chunks, continuing the fma chain s in element order
__device__ __forceinline__ float fma_chain8(const uint4& u, const uint4& v, float s) {
    s = fma_bf16_lo(u.x, v.x, s); s = fma_bf16_hi(u.x, v.x, s);
    s = fma_bf16_lo(u.y, v.y, s); s = fma_bf16_hi(u.y, v.y, s);
    s = fma_bf16_lo(u.z, v.z, s); s = fma_bf16_hi(u.z, v.z, s);
    s = fma_bf16_lo(u.w, v.w, s); s = fma_bf16_hi(u.w, v.w, s);
    return s;
}
// x[0..7] += the 8 bf16 elements of a chunk
__device__ __forceinline__ void add_chunk8(const uint4& u, float* x) {
    x[0] = add_bf16_lo(u.x, x[0]); x[1] = add_bf16_hi(u.x, x[1]);
    x[2] = add_bf16_lo(u.y, x[2]); x[3] = add_bf16_hi(u.y, x[3]);
    x[4] = add_bf16_lo(u.z, x[4]); x[5] = add_bf16_hi(u.z, x[5]);
    x[6] = add_bf16_lo(u.w, x[6]); x[7] = add_bf16_hi(u.w, x[7]);
}

// 16 bytes from global to shared memory without passing through registers; the copies of a
// thread complete in the order of their commit groups
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src_global) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst_smem)), "l"(src_global) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory"); }

// 16 consecutive elements of a row (generic address: shared or global) to fp32
template <typename T>
__device__ __forceinline__ void load16(const T* src, float (&x)[16]) {
    const uint4* v = reinterpret_cast<const uint4*>(src);
    if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint4 w = v[i];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) { x[8 * i + 2 * k] = bf16_lo(ww[k]); x[8 * i + 2 * k + 1] = bf16_hi(ww[k]); }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 w = v[i];
            x[4 * i] = __uint_as_float(w.x); x[4 * i + 1] = __uint_as_float(w.y);
            x[4 * i + 2] = __uint_as_float(w.z); x[4 * i + 3] = __uint_as_float(w.w);
        }
    }
}

template <typename T>
__device__ __forceinline__ void store16(T* dst, const float (&x)[16]) {
    uint4* v = reinterpret_cast<uint4*>(dst);
    if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
            v[i] = make_uint4(pack_bf16x2(x[8 * i], x[8 * i + 1]), pack_bf16x2(x[8 * i + 2], x[8 * i + 3]),
                              pack_bf16x2(x[8 * i + 4], x[8 * i + 5]), pack_bf16x2(x[8 * i + 6], x[8 * i + 7]));
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            v[i] = make_uint4(__float_as_uint(x[4 * i]), __float_as_uint(x[4 * i + 1]),
                              __float_as_uint(x[4 * i + 2]), __float_as_uint(x[4 * i + 3]));
    }
}

// grid: (n_windows + 1, n_chunks, BH); blockIdx.x == n_windows handles the chunk's specials.
template <typename T, bool kTC>
__global__ void __launch_bounds__(kMergeThreads, kTC ? 4 : 3) merge_kernel(MergeArgs a) {
    static_assert(!kTC || sizeof(T) == 2, "the tensor-core matching takes bf16 keys");
    constexpr int VPR = 64 * (int)sizeof(T) / 16;       // 16-byte vectors per row
    constexpr int EPV = 16 / (int)sizeof(T);            // elements per vector
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
    const int tid = threadIdx.x;

    if ((int)blockIdx.x == g.n_windows) {
        // special tokens of the chunk's frames: copied, group size 1
        const long long base = merge_block_base(g, c, -1);
        const int n = nf * g.n_special;
        for (int i = tid; i < n * VPR; i += kMergeThreads) {
            const int k = i / VPR, v = i % VPR;
            const long long t = (long long)(f0 + k / g.n_special) * g.L + k % g.n_special;
            if (!SGA_CHECK_INDEX(base + k, g.M, 22)) continue;
            reinterpret_cast<uint4*>(Xm + (base + k) * 64)[v] = __ldg(reinterpret_cast<const uint4*>(X + t * 64) + v);
            if (Ym) reinterpret_cast<uint4*>(Ym + (base + k) * 64)[v] = __ldg(reinterpret_cast<const uint4*>(Y + t * 64) + v);
        }
        for (int k = tid; k < n; k += kMergeThreads) {
            const long long t = (long long)(f0 + k / g.n_special) * g.L + k % g.n_special;
            if (!SGA_CHECK_INDEX(t, g.T, 20) || !SGA_CHECK_INDEX(base + k, g.M, 22)) continue;
            map[t] = (int32_t)(base + k);
            if (lg) lg[base + k] = 0.f;
        }
        return;
    }

    const int w = blockIdx.x;
    const int ws = merge_window_size(g, w);
    const int nb = nf * ws;                         // tokens of the block: frame-major, then patch
    const int n_src = (nf - 1) * ws;
    const long long r = ((long long)n_src * g.r_permille) / 1000;
    const long long base = merge_block_base(g, c, w);
    const int nb_max = a.nb_max;
    const bool y_smem = a.y_smem && Y;

    extern __shared__ __align__(16) uint8_t smem[];
    T* ys = reinterpret_cast<T*>(smem);                                     // [nb][64] when staged
    float* xs = reinterpret_cast<float*>(smem + (a.y_smem ? nb_max * 64 * (int)sizeof(T) : 0));  // [nb][kXS]
    float* nrm = xs + (kTC ? 0 : nb_max * kXS);                             // [nb]
    float* sim = nrm + nb_max;                                              // partials, then [n_src]
    int* best = reinterpret_cast<int*>(sim + merge_partials(nb_max));      // partials, then [n_src]
    uint32_t* mflag = reinterpret_cast<uint32_t*>(best + merge_partials(nb_max));   // merged-source bits
    // tensor-core path: mbarrier, TMEM address, then the A (sources) and B (destinations) tiles
    uint8_t* tc_misc = reinterpret_cast<uint8_t*>(mflag + (nb_max + 31) / 32);
    tc_misc = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_misc) + 7) & ~uintptr_t(7));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tc_misc + 8);
    uint8_t* tileA = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_misc + 16) + 1023) & ~uintptr_t(1023));
    uint8_t* tileB = tileA + kTcMaxSrc * 128;
    float* inv_nd = reinterpret_cast<float*>(tileB + merge_tc_npad(ws) * 128);   // [ws]: 1 / n_d, or 0
    uint8_t* shortlist = reinterpret_cast<uint8_t*>(inv_nd + kTcMaxDst);        // [kTcList][128]
    const int npad = merge_tc_npad(ws);
    const uint32_t tmem_cols = npad <= 32 ? 32u : npad <= 64 ? 64u : 128u;
    if constexpr (kTC) {
        if (tid < 32) {
            tmem_alloc(smem_u32(tmem_slot), tmem_cols);
            tmem_relinquish();
        }
        if (tid == 0) {
            mbar_init(smem_u32(tc_misc), 1);
            mbar_fence_init();
        }
    }

    // tensor-core path: entry k's row lives only in its bf16 tile (B: destinations, A:
    // sources); 8 dims of 16-byte chunk c, exactly as fp32
    auto tchunk = [&](int k, int c) -> uint4 {                  // the raw 16 bytes
        const int row = k < ws ? k : k - ws;
        const uint8_t* tile = k < ws ? tileB : tileA;
        return *reinterpret_cast<const uint4*>(tile + row * 128 + ((c ^ (row & 7)) << 4));
    };
    auto xchunk = [&](int k, int c, float (&x)[8]) {
        const int row = k < ws ? k : k - ws;
        const uint8_t* tile = k < ws ? tileB : tileA;
        const uint4 v = *reinterpret_cast<const uint4*>(tile + row * 128 + ((c ^ (row & 7)) << 4));
        x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
        x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
    };
    // token of block entry i; its frame i / ws from a float product: i + 1/2 lies at least 1/2
    // from every multiple of ws, and the product's error, under (i / ws + 1) 2^-22, stays below
    // 1 / (2 ws) while nb < 2^20 (a block's rows fit in shared memory)
    const float inv_ws = 1.0f / (float)ws;
    auto tok = [&](int i) -> long long {
        const int fi = (int)(((float)i + 0.5f) * inv_ws);
        return (long long)(f0 + fi) * g.L + g.n_special + (long long)w * g.n_s + (i - fi * ws);
    };
    // 1. the block's rows: X as fp32 (exact), Y as stored.  The tensor-core path copies both
    //    straight into shared memory, X (the bf16 tiles) and Y in two commit groups, so that the
    //    values arrive while the keys are matched.
    if constexpr (kTC) {
        for (int i = tid; i < nb * VPR; i += kMergeThreads) {
            const int k = i / VPR, v = i % VPR;
            const int row = k < ws ? k : k - ws;
            uint8_t* tile = k < ws ? tileB : tileA;
            cp_async16(tile + row * 128 + ((v ^ (row & 7)) << 4), reinterpret_cast<const uint4*>(X + tok(k) * 64) + v);
        }
        cp_async_commit();
        if (y_smem)
            for (int i = tid; i < nb * VPR; i += kMergeThreads) {
                const int k = i / VPR, v = i % VPR;
                cp_async16(reinterpret_cast<uint4*>(ys + k * 64) + v, reinterpret_cast<const uint4*>(Y + tok(k) * 64) + v);
            }
        cp_async_commit();
        cp_async_wait<1>();
    } else {
        for (int i = tid; i < nb * VPR; i += kMergeThreads) {
            const int k = i / VPR, v = i % VPR;
            const long long t = tok(k);
            const uint4 wv = __ldg(reinterpret_cast<const uint4*>(X + t * 64) + v);
            float4* dst = reinterpret_cast<float4*>(xs + k * kXS + v * EPV);
            if constexpr (sizeof(T) == 2) {
                dst[0] = make_float4(bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y));
                dst[1] = make_float4(bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w));
            } else {
                dst[0] = make_float4(__uint_as_float(wv.x), __uint_as_float(wv.y), __uint_as_float(wv.z),
                                     __uint_as_float(wv.w));
            }
            if (y_smem) reinterpret_cast<uint4*>(ys + k * 64)[v] = __ldg(reinterpret_cast<const uint4*>(Y + t * 64) + v);
        }
    }
    if constexpr (kTC) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // 2. norms: sqrt_rn of the fma chain of squares, dimensions in order
    for (int k = tid; k < nb; k += kMergeThreads) {
        float s = 0.f;
        if constexpr (kTC) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 u = tchunk(k, c);
                s = fma_chain8(u, u, s);
            }
        } else {
            const float4* row = reinterpret_cast<const float4*>(xs + k * kXS);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float4 x = row[q];
                s = __fmaf_rn(x.x, x.x, s);
                s = __fmaf_rn(x.y, x.y, s);
                s = __fmaf_rn(x.z, x.z, s);
                s = __fmaf_rn(x.w, x.w, s);
            }
        }
        nrm[k] = __fsqrt_rn(s);
        if (kTC && k < ws) inv_nd[k] = s == 0.f ? 0.f : __frcp_rn(nrm[k]);
    }
    if (kTC && tid >= ws && tid < npad) inv_nd[tid] = __int_as_float(0x7fffffff);
    __syncthreads();
    // 3. every source (entries ws .. nb-1) finds its destination (entries 0 .. ws-1): the first
    //    maximum of cos = dot / (n_a * n_b), each dot an fma chain over the dimensions in order.
    //    The tensor-core path shortlists with one MMA and runs the chains on the shortlist only.
    //    The CUDA-core path splits the destinations into G contiguous groups so that all threads
    //    work; each (source, group) item keeps four dot products in flight, and the groups' first
    //    maxima are combined in ascending order, which gives the first maximum over all
    //    destinations.
    if constexpr (kTC) {
        const uint32_t tmem = *tmem_slot;
        const uint32_t bar = smem_u32(tc_misc);
        if (tid == 0 && n_src > 0) {
            const uint64_t dA = smem_desc_sw128(smem_u32(tileA), 16);
            const uint64_t dB = smem_desc_sw128(smem_u32(tileB), 16);
            const uint32_t idesc = idesc_bf16_f32(128, npad, false);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_ss(tmem, dA + 2 * kk, dB + 2 * kk, idesc, kk > 0 ? 1u : 0u);
            mma_commit(bar);
        }
        if (tid < 128 && n_src > 0) {
            // one thread per source (TMEM lane); the wait is bounded
            const long long t0 = clock64();
            while (!mbar_try_wait(bar, 0)) {
                if (clock64() - t0 > kTimeoutCycles) {
                    atomicExch(&g_status, (int)SGA_ERR_TIMEOUT);
                    break;
                }
            }
            tc_fence_after();
            const int a2 = tid;
            const bool live = a2 < n_src;
            const uint32_t taddr = tmem + ((uint32_t)(tid & ~31) << 16);
            const float nk = live ? nrm[ws + a2] : 0.f;
            // pass 1: the best approximate cosine, scaled by n_k (the TMEM sum times 1 / n_d)
            float amax = -INFINITY;
            for (int c0 = 0; c0 < npad; c0 += 16) {
                uint32_t r16[16];
                tmem_ld16(taddr + c0, r16);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) amax = fmaxf(amax, __fmul_rn(__uint_as_float(r16[i]), inv_nd[c0 + i]));
            }
            // pass 2: the destinations within the window, in ascending order, onto the source's
            // shortlist; the exact chains run after it, with the warp's lanes together
            const float thr = amax - kMatchWindow * nk;
            int n_cand = 0;
            for (int c0 = 0; c0 < npad; c0 += 16) {
                uint32_t r16[16];
                tmem_ld16(taddr + c0, r16);
                tmem_wait_ld();
                uint32_t cand = 0;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    cand |= __fmul_rn(__uint_as_float(r16[i]), inv_nd[c0 + i]) >= thr ? 1u << i : 0u;
                if (!live) cand = 0;
                for (; cand; cand &= cand - 1) {
                    if (n_cand < kTcList) shortlist[n_cand * kTcMaxSrc + a2] = (uint8_t)(c0 + __ffs(cand) - 1);
                    ++n_cand;
                }
            }
            // the exact cosine of each candidate; the first maximum decides.  A shortlist that
            // overflowed (near-equal destinations) goes on with every destination after its last
            // entry: a superset of the candidates, and every destination that could reach the
            // maximum is a candidate, so the first maximum is the same.
            float bs = -INFINITY;
            int bd = -1;
            const uint8_t* row_a = tileA + a2 * 128;
            auto verify = [&](int d) {
                const float den = __fmul_rn(nk, nrm[d]);
                const uint8_t* row_d = tileB + d * 128;
                float dot = 0.f;
#pragma unroll 2
                for (int c = 0; c < 8; ++c) {
                    const uint4 u = *reinterpret_cast<const uint4*>(row_a + ((c ^ (a2 & 7)) << 4));
                    const uint4 v = *reinterpret_cast<const uint4*>(row_d + ((c ^ (d & 7)) << 4));
                    dot = fma_chain8(u, v, dot);
                }
                const float cs = den == 0.f ? 0.f : __fdiv_rn(dot, den);
                if (cs > bs) { bs = cs; bd = d; }
            };
            const int d_last = n_cand > kTcList ? shortlist[(kTcList - 1) * kTcMaxSrc + a2] : ws - 1;
            const int n_ver = n_cand > kTcList ? kTcList + (ws - 1 - d_last) : n_cand;
            for (int k = 0; k < n_ver; ++k)
                verify(k < kTcList ? shortlist[k * kTcMaxSrc + a2] : d_last + 1 + (k - kTcList));
            if (live) {
                sim[a2] = bs;
                best[a2] = bd;
            }
        }
        tc_fence_before();
        __syncthreads();
    } else {
    const int G = n_src > 0 ? max(1, min(4, kMergeThreads / n_src)) : 1;
    for (int it = tid; it < n_src * G; it += kMergeThreads) {
        const int a2 = it % n_src, grp = it / n_src;
        const int k = ws + a2;
        const int d_beg = (grp * ws) / G, d_end = ((grp + 1) * ws) / G;
        float xk[64];                                            // the source row, in registers
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float4 x = reinterpret_cast<const float4*>(xs + k * kXS)[q];
            xk[4 * q] = x.x; xk[4 * q + 1] = x.y; xk[4 * q + 2] = x.z; xk[4 * q + 3] = x.w;
        }
        const float nk = nrm[k];
        float bs = -INFINITY;
        int bd = -1;
        for (int d0 = d_beg; d0 < d_end; d0 += 4) {
            const int d1 = min(d0 + 1, d_end - 1), d2 = min(d0 + 2, d_end - 1), d3 = min(d0 + 3, d_end - 1);
            float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
            const float4* r0 = reinterpret_cast<const float4*>(xs + d0 * kXS);
            const float4* r1 = reinterpret_cast<const float4*>(xs + d1 * kXS);
            const float4* r2 = reinterpret_cast<const float4*>(xs + d2 * kXS);
            const float4* r3 = reinterpret_cast<const float4*>(xs + d3 * kXS);
#pragma unroll
            for (int q = 0; q < 16; ++q) {                       // dimensions 4q .. 4q+3, in order
                const float4 b0 = r0[q], b1 = r1[q], b2 = r2[q], b3 = r3[q];
                p0 = __fmaf_rn(xk[4 * q], b0.x, p0); p0 = __fmaf_rn(xk[4 * q + 1], b0.y, p0);
                p0 = __fmaf_rn(xk[4 * q + 2], b0.z, p0); p0 = __fmaf_rn(xk[4 * q + 3], b0.w, p0);
                p1 = __fmaf_rn(xk[4 * q], b1.x, p1); p1 = __fmaf_rn(xk[4 * q + 1], b1.y, p1);
                p1 = __fmaf_rn(xk[4 * q + 2], b1.z, p1); p1 = __fmaf_rn(xk[4 * q + 3], b1.w, p1);
                p2 = __fmaf_rn(xk[4 * q], b2.x, p2); p2 = __fmaf_rn(xk[4 * q + 1], b2.y, p2);
                p2 = __fmaf_rn(xk[4 * q + 2], b2.z, p2); p2 = __fmaf_rn(xk[4 * q + 3], b2.w, p2);
                p3 = __fmaf_rn(xk[4 * q], b3.x, p3); p3 = __fmaf_rn(xk[4 * q + 1], b3.y, p3);
                p3 = __fmaf_rn(xk[4 * q + 2], b3.z, p3); p3 = __fmaf_rn(xk[4 * q + 3], b3.w, p3);
            }
            const float dots[4] = {p0, p1, p2, p3};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int d = d0 + q;
                if (d < d_end) {
                    const float den = __fmul_rn(nk, nrm[d]);
                    const float cs = den == 0.f ? 0.f : __fdiv_rn(dots[q], den);
                    if (cs > bs) { bs = cs; bd = d; }
                }
            }
        }
        sim[grp * n_src + a2] = bs;
        best[grp * n_src + a2] = bd;
    }
    __syncthreads();
    if (G > 1) {
        // slot a2 (group 0) is read and then written by thread a2 alone
        for (int a2 = tid; a2 < n_src; a2 += kMergeThreads) {
            float bs = sim[a2];
            int bd = best[a2];
            for (int grp = 1; grp < G; ++grp)
                if (sim[grp * n_src + a2] > bs) { bs = sim[grp * n_src + a2]; bd = best[grp * n_src + a2]; }
            sim[a2] = bs;
            best[a2] = bd;
        }
        __syncthreads();
    }
    }
    // 4. merged sources: the r largest similarities (ties: lower token index = lower entry index,
    //    since entries are in token order); one flag bit per source, a warp's 32 in one word
    for (int a0 = 0; a0 < n_src; a0 += kMergeThreads) {
        const int a2 = a0 + tid;
        bool merged = false;
        if (a2 < n_src) {
            const float sa = sim[a2];
            int ahead = 0;
            for (int b2 = 0; b2 < n_src; ++b2) {
                const float sb = sim[b2];
                ahead += (sb > sa || (sb == sa && b2 < a2)) ? 1 : 0;
            }
            merged = ahead < r;
        }
        const uint32_t bal = __ballot_sync(0xffffffffu, merged);
        const int w0 = a0 + (tid & ~31);
        if ((tid & 31) == 0 && w0 < n_src) mflag[w0 >> 5] = bal;
    }
    if constexpr (kTC) {
        cp_async_wait<0>();                                  // this thread's value rows
        if (tid < 32) {
            tc_fence_after();
            tmem_dealloc(*tmem_slot, tmem_cols);             // the TMEM reads ended before phase 4
        }
    }
    __syncthreads();
    // 5. kept entries get consecutive merged indices in entry (= token) order: the destinations
    //    (entries 0 .. ws-1, never merged) keep their entry index, a kept source loses one for
    //    every merged source before it
    auto is_merged = [&](int a2) -> bool { return (mflag[a2 >> 5] >> (a2 & 31)) & 1u; };
    auto kept_index = [&](int k) -> int {
        if (k < ws) return k;
        const int a2 = k - ws;
        int before = __popc(mflag[a2 >> 5] & ((1u << (a2 & 31)) - 1u));
        for (int q = 0; q < (a2 >> 5); ++q) before += __popc(mflag[q]);
        return k - before;
    };
    // 8. group means of the kept entries (a destination plus the sources merged into it, summed
    //    in entry order), 16 dimensions per work item, and ln of the group size
    int* cnt = reinterpret_cast<int*>(sim);                  // [ws]: count, then running position
    int* list = cnt + ws;                                   // [n_src] members, destination-major
    auto mean_item = [&](int k, int e0) {
        const long long mi = base + kept_index(k);
        if (!SGA_CHECK_INDEX(mi, g.M, 21)) return;
        float sx[16], sy[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) sy[e] = 0.f;
        if constexpr (kTC) {
            float x8[8];
            xchunk(k, e0 >> 3, x8);
#pragma unroll
            for (int e = 0; e < 8; ++e) sx[e] = x8[e];
            xchunk(k, (e0 >> 3) + 1, x8);
#pragma unroll
            for (int e = 0; e < 8; ++e) sx[8 + e] = x8[e];
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) sx[e] = xs[k * kXS + e0 + e];
        }
        if (Y) load16<T>(y_smem ? ys + k * 64 + e0 : Y + tok(k) * 64 + e0, sy);
        int cntk = 1;
        if (k < ws) {
            const int m_end = cnt[k], m_beg = k > 0 ? cnt[k - 1] : 0;
            cntk += m_end - m_beg;
            for (int q = m_beg; q < m_end; ++q) {
                const int ks = ws + list[q];
                if constexpr (kTC) {
                    add_chunk8(tchunk(ks, e0 >> 3), sx);
                    add_chunk8(tchunk(ks, (e0 >> 3) + 1), sx + 8);
                    if (Y) {
                        const uint4* yr = reinterpret_cast<const uint4*>(y_smem ? ys + ks * 64 + e0 : Y + tok(ks) * 64 + e0);
                        add_chunk8(yr[0], sy);
                        add_chunk8(yr[1], sy + 8);
                    }
                    continue;
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) sx[e] += xs[ks * kXS + e0 + e];
                }
                if (Y) {
                    float ty[16];
                    load16<T>(y_smem ? ys + ks * 64 + e0 : Y + tok(ks) * 64 + e0, ty);
#pragma unroll
                    for (int e = 0; e < 16; ++e) sy[e] += ty[e];
                }
            }
        }
        const float inv = 1.0f / (float)cntk;
#pragma unroll
        for (int e = 0; e < 16; ++e) { sx[e] *= inv; sy[e] *= inv; }
        store16<T>(Xm + mi * 64 + e0, sx);
        if (Ym) store16<T>(Ym + mi * 64 + e0, sy);
        if (lg && e0 == 0) lg[mi] = logf((float)cntk);
    };
    if (tid < 32) {
        // 7. each destination's merged sources, in ascending entry order: counted, offsets
        //    scanned and listed by one warp, 32 sources at a time (the lanes of one destination
        //    find each other with a match), so the group sums run over the members alone and in
        //    the same order as before.  The lists reuse the similarity array (ws + n_src = nb
        //    entries).  The other warps meanwhile write the map and the kept sources' rows.
        const int lane = tid;
        for (int d = lane; d < ws; d += 32) cnt[d] = 0;
        __syncwarp();
        for (int c0 = 0; c0 < n_src; c0 += 32) {
            const int a2 = c0 + lane;
            const bool mg = a2 < n_src && is_merged(a2);
            const int d = mg ? best[a2] : -1;
            const uint32_t m = __match_any_sync(0xffffffffu, d);
            if (mg && lane == __ffs(m) - 1) cnt[d] += __popc(m);
            __syncwarp();
        }
        // exclusive scan of the counts: cnt[d] becomes the first list position of d
        int run = 0;
        for (int d0 = 0; d0 < ws; d0 += 32) {
            const int d = d0 + lane;
            const int v = d < ws ? cnt[d] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (d < ws) cnt[d] = run + incl - v;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        __syncwarp();
        for (int c0 = 0; c0 < n_src; c0 += 32) {
            const int a2 = c0 + lane;
            const bool mg = a2 < n_src && is_merged(a2);
            const int d = mg ? best[a2] : -1;
            const uint32_t m = __match_any_sync(0xffffffffu, d);
            if (mg) list[cnt[d] + __popc(m & ((1u << lane) - 1u))] = a2;
            __syncwarp();
            if (mg && lane == __ffs(m) - 1) cnt[d] += __popc(m);
            __syncwarp();
        }
        // now cnt[d] is one past the last member of d; its first is cnt[d - 1] (0 for d = 0)
    } else {
        // 6. map: every token to its merged row (a merged source to its destination's, whose
        //    merged index is its entry index)
        for (int k = tid - 32; k < nb; k += kMergeThreads - 32) {
            const long long mi = base + (k >= ws && is_merged(k - ws) ? best[k - ws] : kept_index(k));
            if (SGA_CHECK_INDEX(tok(k), g.T, 20) && SGA_CHECK_INDEX(mi, g.M, 21)) map[tok(k)] = (int32_t)mi;
        }
        // 8a. the kept sources' rows (groups of one): the mean of one row is the row itself, so
        //    the tensor-core path copies its 16-byte chunks (and ln 1 = 0)
        if constexpr (kTC) {
            for (int it = tid - 32; it < n_src * VPR; it += kMergeThreads - 32) {
                const int a2 = it / VPR, v = it % VPR;
                if (is_merged(a2)) continue;
                const int k = ws + a2;
                const long long mi = base + kept_index(k);
                if (!SGA_CHECK_INDEX(mi, g.M, 21)) continue;
                reinterpret_cast<uint4*>(Xm + mi * 64)[v] = tchunk(k, v);
                if (Ym)
                    reinterpret_cast<uint4*>(Ym + mi * 64)[v] =
                        y_smem ? reinterpret_cast<const uint4*>(ys + k * 64)[v]
                               : __ldg(reinterpret_cast<const uint4*>(Y + tok(k) * 64) + v);
                if (lg && v == 0) lg[mi] = 0.f;
            }
        } else {
            for (int it = tid - 32; it < n_src * 4; it += kMergeThreads - 32) {
                const int k = ws + (it >> 2);
                if (!is_merged(k - ws)) mean_item(k, (it & 3) * 16);
            }
        }
    }
    __syncthreads();
    // 8b. the destinations' group means
    for (int it = tid; it < ws * 4; it += kMergeThreads) mean_item(it >> 2, (it & 3) * 16);
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
    const int32_t mi = __ldg(map + row);
    if (!SGA_CHECK_INDEX(mi, M, 23)) return;
    const long long src = bh * M + mi;
    reinterpret_cast<uint4*>(Y)[row * kVec + v] = __ldg(reinterpret_cast<const uint4*>(Ym) + src * kVec + v);
}

}  // namespace sga
