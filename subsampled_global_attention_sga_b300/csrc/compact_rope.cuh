// compact_rope.cuh -- the SGA compaction step with the 2D rotary embedding fused (bf16): one
// streaming pass over K and V that rotates every key, copies the kept rows into contiguous
// K_S / V_S and sums the dropped rows.
//
// "AVGGT: Rethinking Global Attention for Accelerating VGGT", Key design 2 (K and V replaced by
// their subset S) and Key design 3 (one mean key/value stands for all dropped patches); "HTTM:
// Head-wise Temporal Token Merging for Faster VGGT", section 3 (VGGT rotates Q and K in every
// layer, so the compacted keys are the rotated ones).
//
// HBM-bound, and the rotation adds enough per-row work that loads issued by the computing threads
// themselves leave too few bytes in flight.  So the loads are decoupled: a producer warp streams
// 64-row stages of K and V (plus the 64 slot entries) into a ring of shared-memory buffers with
// TMA (128-byte swizzle, so that the 8 rows a warp reads at once sit in distinct banks), and 8
// consumer warps rotate, store or sum.  CTAs are persistent (two per SM) and walk fixed work
// items of rows_per_chunk rows of one (batch, head); each item's partial sums are reduced in a
// fixed order and written to its own slot of the scratch buffer, as in the plain kernel.
#pragma once

#include "compact.cuh"

namespace sga {
namespace cr {

constexpr int kStageRows = 64;
constexpr int kStages = 6;
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;          // + one producer warp
constexpr int kTileBytes = kStageRows * 128;                  // 64 rows x 64 bf16
constexpr int kSlotBytes = kStageRows * 4;
// shared memory (offsets from a 1024-byte aligned base): K and V tiles of every stage, the slot
// entries of every stage, barriers + abort flag, the reduction buffer, the (cos, sin) table
constexpr int OFF_KV = 0;
constexpr int OFF_SLOT = OFF_KV + kStages * 2 * kTileBytes;
constexpr int OFF_BAR = OFF_SLOT + kStages * kSlotBytes;
constexpr int OFF_RED = OFF_BAR + 2 * kStages * 8 + 16;
constexpr int kRedFloats = kConsumerWarps * 4 * 32;          // [warp][lane group][16 key + 16 value sums]
constexpr int OFF_TAB = OFF_RED + kRedFloats * 4;
__host__ __device__ constexpr size_t smem_bytes(int rope_P) {
    return (size_t)OFF_TAB + (size_t)rope_P * kRopeTabStride * sizeof(float2) + 1024;
}

struct Args {
    long long T;            // tokens per (batch, head)
    long long S;            // kept tokens per (batch, head)
    int rows_per_chunk;     // rows of one work item (a multiple of kStageRows)
    int n_chunks;           // work items per (batch, head)
    long long n_items;      // BH * n_chunks
    __nv_bfloat16* KS;
    __nv_bfloat16* VS;
    float* partials;        // [BH, n_chunks, 128]
    RopeArgs rope;
    const int32_t* slot;    // the plan's slot table, padded to a multiple of 64 entries
};

// plain bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// tmK, tmV: 3-D maps over [BH, T, 64] bf16, box 64 x 64 rows, 128-byte swizzle, zero fill past T.
__global__ void __launch_bounds__(kThreads, 2)
compact_rope_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(base);
    auto full = [&](int s) -> uint32_t { return sbase + OFF_BAR + 8 * s; };
    auto empty = [&](int s) -> uint32_t { return sbase + OFF_BAR + 8 * (kStages + s); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + OFF_BAR + 16 * kStages);
    float* red = reinterpret_cast<float*>(base + OFF_RED);
    float2* tab = reinterpret_cast<float2*>(base + OFF_TAB);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kConsumerWarps);
        }
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    for (int i = threadIdx.x; i < a.rope.P * 16; i += kThreads)
        tab[(i >> 4) * kRopeTabStride + (i & 15)] = a.rope.tab[i];
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------------ producer
        uint32_t it = 0, issued = 0;
        bool ok = true;
        for (long long item = blockIdx.x; item < a.n_items && ok; item += gridDim.x) {
            const int bh = (int)(item / a.n_chunks);
            const long long r_begin = (item % a.n_chunks) * (long long)a.rows_per_chunk;
            const long long r_end = r_begin + a.rows_per_chunk < a.T ? r_begin + a.rows_per_chunk : a.T;
            for (long long r0 = r_begin; r0 < r_end; r0 += kStageRows, ++it) {
                const int st = (int)(it % kStages);
                if (!__all_sync(0xffffffffu, mbar_wait(empty(st), ((it / kStages) & 1) ^ 1, abort_flag))) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    const uint32_t kdst = sbase + OFF_KV + st * 2 * kTileBytes;
                    mbar_arrive_expect_tx(full(st), 2 * kTileBytes + kSlotBytes);
                    tma_load_3d(kdst, &tmK, full(st), 0, (int)r0, bh);
                    tma_load_3d(kdst + kTileBytes, &tmV, full(st), 0, (int)r0, bh);
                    bulk_load(sbase + OFF_SLOT + st * kSlotBytes, a.slot + r0, kSlotBytes, full(st));
                }
                __syncwarp();
                issued = it + 1;
            }
        }
        if (!ok) {
            // let the copies already issued land before the CTA leaves
            const long long t0 = clock64();
            for (uint32_t i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
                while (!mbar_try_wait(full((int)(i % kStages)), (i / kStages) & 1))
                    if (clock64() - t0 > kTimeoutCycles / 8) break;
        }
    } else {
        // ------------------------------------------------------------------ consumers
        // Lane l of warp w takes row 8w + (l mod 8) of each stage and, with g = l / 8, the two
        // 16-byte vectors va = (g mod 2) + 4 (g / 2) and va + 2 of it: dims d0..d0+7 and
        // d0+16..d0+23 of one 32-dim half, which rotate together.  The 8 lanes of a shared-memory
        // phase read one vector of 8 consecutive rows: distinct banks under the swizzle.
        const int rr = warp * 8 + (lane & 7);
        const int g = lane >> 3;
        const int va = (g & 1) + 4 * (g >> 1);
        const int d0 = va * 8;
        const int L = a.rope.L, ns = a.rope.n_special, gw = a.rope.grid_w, off = a.rope.pos_offset;
        const float inv_gw = 1.0f / (float)gw;
        const int step_mod = kStageRows % L;
        uint32_t it = 0;
        bool ok = true;
        for (long long item = blockIdx.x; item < a.n_items; item += gridDim.x) {
            const int bh = (int)(item / a.n_chunks);
            const long long r_begin = (item % a.n_chunks) * (long long)a.rows_per_chunk;
            const long long r_end = r_begin + a.rows_per_chunk < a.T ? r_begin + a.rows_per_chunk : a.T;
            uint4* KS = reinterpret_cast<uint4*>(a.KS) + (long long)bh * a.S * 8;
            uint4* VS = reinterpret_cast<uint4*>(a.VS) + (long long)bh * a.S * 8;
            float ks[16], vs[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) { ks[e] = 0.f; vs[e] = 0.f; }
            int pos = (int)((r_begin + rr) % L);                 // token position within its frame
            for (long long r0 = r_begin; r0 < r_end; r0 += kStageRows, ++it) {
                const int st = (int)(it % kStages);
                // after a failure every wait returns at once: the warps still meet at the barriers
                ok = __all_sync(0xffffffffu, mbar_wait(full(st), (it / kStages) & 1, abort_flag)) && ok;
                const long long t = r0 + rr;
                if (ok && t < r_end) {
                    const int sl = reinterpret_cast<const int*>(base + OFF_SLOT + st * kSlotBytes)[rr];
                    const uint8_t* krow = base + OFF_KV + st * 2 * kTileBytes + rr * 128;
                    const uint8_t* vrow = krow + kTileBytes;
                    const int sw = rr & 7;
                    const uint4 ka = *reinterpret_cast<const uint4*>(krow + ((va ^ sw) << 4));
                    const uint4 kb = *reinterpret_cast<const uint4*>(krow + (((va + 2) ^ sw) << 4));
                    const uint4 wa = *reinterpret_cast<const uint4*>(vrow + ((va ^ sw) << 4));
                    const uint4 wb = *reinterpret_cast<const uint4*>(vrow + (((va + 2) ^ sw) << 4));
                    int pr = 0, pc = 0;
                    if (pos >= ns) {
                        // grid row from a float quotient, exact for q < 2^21 (the table bounds
                        // the grid far below that)
                        const int q = pos - ns;
                        const int qr = (int)(((float)q + 0.5f) * inv_gw);
                        pr = qr + off;
                        pc = q - qr * gw + off;
                    }
                    const float2* tb = tab + ((d0 & 32) ? pc : pr) * kRopeTabStride + (d0 & 15);
                    float x0[8], x1[8];
                    Vec16<__nv_bfloat16>::unpack(ka, x0);
                    Vec16<__nv_bfloat16>::unpack(kb, x1);
                    float4 cs4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) cs4[e] = reinterpret_cast<const float4*>(tb)[e];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {                  // dims d0+e and d0+e+16
                        const float2 cs = (e & 1) ? make_float2(cs4[e >> 1].z, cs4[e >> 1].w)
                                                  : make_float2(cs4[e >> 1].x, cs4[e >> 1].y);
                        const float y0 = fmaf(-x1[e], cs.y, x0[e] * cs.x);
                        const float y1 = fmaf(x0[e], cs.y, x1[e] * cs.x);
                        x0[e] = y0;
                        x1[e] = y1;
                    }
                    if (sl >= 0) {
                        if (SGA_CHECK_INDEX(sl, a.S, 3)) {
                            uint4* ksr = KS + (long long)sl * 8;
                            uint4* vsr = VS + (long long)sl * 8;
                            ksr[va] = Vec16<__nv_bfloat16>::pack(x0);
                            ksr[va + 2] = Vec16<__nv_bfloat16>::pack(x1);
                            vsr[va] = wa;
                            vsr[va + 2] = wb;
                        }
                    } else {
                        float v0[8], v1[8];
                        Vec16<__nv_bfloat16>::unpack(wa, v0);
                        Vec16<__nv_bfloat16>::unpack(wb, v1);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            ks[e] += x0[e];
                            ks[8 + e] += x1[e];
                            vs[e] += v0[e];
                            vs[8 + e] += v1[e];
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty(st));
                pos += step_mod;
                if (pos >= L) pos -= L;
            }
            // the item's sums: over the 8 rows of the warp (fixed shuffle tree), then over the
            // warps in order
#pragma unroll
            for (int e = 0; e < 16; ++e) {
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    ks[e] += __shfl_xor_sync(0xffffffffu, ks[e], o);
                    vs[e] += __shfl_xor_sync(0xffffffffu, vs[e], o);
                }
            }
            if ((lane & 7) == 0) {
                float* rw = red + (warp * 4 + g) * 32;
#pragma unroll
                for (int e = 0; e < 16; ++e) { rw[e] = ks[e]; rw[16 + e] = vs[e]; }
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");
            if (threadIdx.x < 128) {
                // output j: dim j of the key sum (j < 64) or of the value sum; vector v = dim / 8
                // is held by lane group (v mod 2) + 2 (v / 4), as its first (v mod 4 < 2) or
                // second vector
                const int which = threadIdx.x >> 6, dim = threadIdx.x & 63;
                const int v = dim >> 3, w4 = v & 3;
                const int gg = (w4 & 1) + 2 * (v >> 2);
                const int e = (w4 >> 1) * 8 + (dim & 7);
                float s = 0.f;
                for (int w = 0; w < kConsumerWarps; ++w) s += red[(w * 4 + gg) * 32 + which * 16 + e];
                a.partials[item * 128 + threadIdx.x] = s;
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");
        }
    }
}

}  // namespace cr
}  // namespace sga
