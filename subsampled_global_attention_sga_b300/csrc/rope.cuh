// rope.cuh -- 2D rotary position embedding of Q and K rows (d = 64), fused into the SGA layer.
//
// VGGT re-applies rotary position encoding in every layer ("HTTM: Head-wise Temporal Token
// Merging for Faster VGGT", section 3).  The pages give no convention; the one used: head dims
// [0, 32) rotate by the token's row position, [32, 64) by its column position; in each half the
// pairs (j, j+16), j < 16, rotate by the angle pos * base^(-j/16); a patch (r, c) sits at
// (r + pos_offset, c + pos_offset) and the camera/register tokens at position 0 (unrotated).
// The cos/sin table (positions x 16 frequencies) is computed in double on the host.
#pragma once

#include "common.cuh"

namespace sga {

struct RopeArgs {
    int on;                 // 0: no rotation
    const float2* tab;      // [P][16] (cos, sin) of pos * base^(-j/16)
    int P;                  // positions in the table
    int L, n_special, grid_w, pos_offset;
};

// (row, column) position of token t (index within one (batch, head) sequence)
__device__ __forceinline__ void rope_pos(const RopeArgs& a, long long t, int& pr, int& pc) {
    const int p = (int)t % a.L;             // token indices of a sequence are below 2^31
    if (p < a.n_special) {
        pr = 0;
        pc = 0;
    } else {
        const int q = p - a.n_special;
        pr = q / a.grid_w + a.pos_offset;
        pc = q % a.grid_w + a.pos_offset;
    }
}

// Rotate a full 64-wide row held in registers (fp32), table read from global memory.
__device__ __forceinline__ void rope_row64(const RopeArgs& a, long long t, float (&x)[64]) {
    int pos[2];
    rope_pos(a, t, pos[0], pos[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float2* tb = a.tab + pos[h] * 16;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float2 cs = __ldg(tb + j);
            const float x0 = x[32 * h + j], x1 = x[32 * h + j + 16];
            x[32 * h + j] = x0 * cs.x - x1 * cs.y;
            x[32 * h + j + 16] = x0 * cs.y + x1 * cs.x;
        }
    }
}

}  // namespace sga

namespace sga {

// In-place rotation of X [rows_total, 64] (rows_total = B*H*T_seq): one thread per row.
// Plain loads (not the read-only path): each row is written back by the thread that read it.
template <typename T>
__global__ void __launch_bounds__(256) rope2d_kernel(T* X, long long rows_total, long long T_seq, RopeArgs a) {
    const long long row = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= rows_total) return;
    T* xr = X + row * 64;
    float x[64];
    if constexpr (sizeof(T) == 2) {
        const uint4* p = reinterpret_cast<const uint4*>(xr);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 v = p[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) { x[8 * i + 2 * k] = bf16_lo(w[k]); x[8 * i + 2 * k + 1] = bf16_hi(w[k]); }
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(xr);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float4 v = p[i];
            x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
        }
    }
    rope_row64(a, row % T_seq, x);
    if constexpr (sizeof(T) == 2) {
        uint4* p = reinterpret_cast<uint4*>(xr);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            p[i] = make_uint4(pack_bf16x2(x[8 * i], x[8 * i + 1]), pack_bf16x2(x[8 * i + 2], x[8 * i + 3]),
                              pack_bf16x2(x[8 * i + 4], x[8 * i + 5]), pack_bf16x2(x[8 * i + 6], x[8 * i + 7]));
    } else {
        float4* p = reinterpret_cast<float4*>(xr);
#pragma unroll
        for (int i = 0; i < 16; ++i) p[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
    }
}

}  // namespace sga
