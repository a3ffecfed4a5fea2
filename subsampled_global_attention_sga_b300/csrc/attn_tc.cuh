// attn_tc.cuh -- tensor-core attention kernel for sm_103a (bf16 in, fp32 accumulate):
// TMA-staged tiles, tcgen05.mma with accumulators in Tensor Memory, online softmax on the
// CUDA cores, persistent CTAs.  One kernel serves SGA (keys = the compacted K_S/V_S, plus the
// diagonal and mean components folded into each row's running max and sum), dense global
// attention and frame-local attention (keys = one frame).
//
// Sources: "AVGGT: Rethinking Global Attention for Accelerating VGGT", Key design 2 (attention
// softmax(QK^T/sqrt(d))V over the kept set, all queries kept) and Key design 3 (the diagonal
// and mean components share the softmax); "RegimeVGGT ...", Key design 2 (ln g logit bias).
//
// Work unit: two 128-row query tiles of one segment (a (batch, head) pair, or one frame of it)
// against all key tiles of that segment; a segment with an odd tile count leaves its last tile to
// a mixed unit with the next segment's (each tile against its own segment's keys).  A unit is a
// sequence of slots n = 2j + t (query tile t, key tile j); a CTA numbers the slots of its units
// on from one unit to the next.  Roles (384 threads):
//   warp 0      TMA producer: the two Q tiles of a unit (into one of two Q buffers, so the next
//               unit's are in place before this one ends), then a STAGES-deep ring of K and V
//               tiles (one barrier pair per stage)
//   warps 1, 2  MMA issuers (one elected lane each), taking turns:
//                 S(n)  = Q_t K_j^T  (M=128, N=128, K=64; A, B from shared memory)
//                 O_t  += P(n) V_j   (M=128, N=64,  K=128; P from TMEM, V from shared memory)
//               batch G_n = PV(n), then QK(n + 3) (possibly of the next unit); issuer n mod 2
//               issues it once P(n) is ready
//   warps 4-7   softmax + epilogue of query tile 0 (one thread per row)
//   warps 8-11  softmax + epilogue of query tile 1
// TMEM columns: O_0 [0,64) O_1 [64,128), and three S buffers [128,256) [256,384) [384,512).  The
// S of global slot n goes to buffer n mod 3 and its P (bf16 pairs) is written over the first 64
// columns of that S.  PV(n) frees the buffer that QK(n + 3) then fills, so each softmax
// warpgroup finds its next S computed while it works: the tensor pipe and the softmax warps no
// longer wait on each other tile by tile.
// With a per-key bias (size-aware attention, "RegimeVGGT ..." Key design 2: a key standing
// for g tokens carries the logit bias ln g), QK^T gets a fifth K = 16 step: the Q side is a
// constant block with ones in columns 0-1, the K side holds bias/scale split into a bf16 high
// and low part in columns 0-1 (written by the producer warp from the fp32 bias), so the
// accumulator already contains q.k + bias/scale and the softmax is unchanged.
// A row's reference max is only moved (and O rescaled in TMEM) when its logits exceed it by
// more than 2^8; the final normalisation uses the same reference, so the result is exact either
// way.  The exponentials are taken against the current reference first; a tile sum above 2^7
// sends the tile to the max-first decision, so the row maximum is off the per-tile path.
#pragma once

#include "extras.cuh"

namespace sga {
namespace tc {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int HD = 64;
constexpr int STAGES = 4;
constexpr int TILE_BYTES = BM * HD * 2;        // one 128 x 64 bf16 tile = 16 KB
constexpr int NUM_THREADS = 384;
constexpr uint32_t TMEM_COLS = 512;
__host__ __device__ constexpr uint32_t col_o(int t) { return 64u * (uint32_t)t; }            // O_t
__host__ __device__ constexpr uint32_t col_buf(uint32_t b) { return 128u + 128u * b; }     // S (then P) buffer b
constexpr uint32_t NUM_SBUF = 3;
constexpr float kRescaleThreshold = 8.0f;      // base-2: rescale when the max grows by > 2^8
constexpr float kSumTrigger = 128.0f;          // a tile sum above this takes the max-first decision

// Register split (setmaxnreg): the kernel is launched with LAUNCH_REGS per thread; warpgroup 0
// (TMA producer, two MMA issuers, one idle warp) gives registers back, the two softmax warpgroups
// take them.  The split must add up to the launch total, otherwise setmaxnreg.inc cannot be
// satisfied; the host checks the compiled register count before every launch.
constexpr uint32_t LAUNCH_REGS = 168;
constexpr uint32_t REGS_CTRL = 72;
constexpr uint32_t REGS_SOFTMAX = 216;
static_assert(REGS_CTRL * 128 + REGS_SOFTMAX * 256 == LAUNCH_REGS * NUM_THREADS, "register split");
static_assert(LAUNCH_REGS * NUM_THREADS <= 65536, "register file");

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + 4 * TILE_BYTES;          // Q: two buffers of two tiles
constexpr int OFF_V = OFF_K + STAGES * TILE_BYTES;
// bias blocks: 128 rows x 16 bf16 columns in the no-swizzle K-major core-matrix layout
// (8 rows x 16 bytes per core matrix; LBO = 128 B between the two K halves, SBO = 256 B
// between groups of 8 rows)
constexpr int EXT_BYTES = 128 * 16 * 2;
constexpr int OFF_QEXT = OFF_V + STAGES * TILE_BYTES;
constexpr int OFF_KEXT = OFF_QEXT + EXT_BYTES;
constexpr int OFF_BAR = OFF_KEXT + STAGES * EXT_BYTES;
// barriers: q_full[2], q_empty[2], kv_full[S], kv_empty[S], s_full[3], p_ready[3], o_done[2],
//           o_free[2], drain, q_rot[2], pv_done[2], turn[2]
constexpr int NUM_BARS = 4 + 2 * STAGES + 6 + 4 + 1 + 2 + 2 + 2;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
// a softmax thread's row state while its unit waits for the epilogue: 8 words per thread, stored
// word-major ([word][thread]) so that a warp's accesses fall in distinct banks
constexpr int OFF_PEND = OFF_MISC + 16;
constexpr int PEND_WORDS = 8;
constexpr int SMEM_BYTES = OFF_PEND + PEND_WORDS * 256 * 4 + 1024;   // + alignment slack

constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, HD, true);

struct TcArgs {
    int n_seg;              // segments
    int seg_rows;           // query rows per segment
    int kv_rows;            // keys per segment
    int n_pairs;            // full pairs of 128-row query tiles per segment (q_tiles / 2)
    int n_kv_tiles;         // ceil(kv_rows / 128)
    long long n_units;      // n_seg * n_pairs, + ceil(n_seg / 2) mixed units when q_tiles is odd
    int group;              // with mixed units: units per pair of segments (2 n_pairs + 1); else 0
    int last_row0;          // first row of a segment's last query tile ((q_tiles - 1) * 128)
    float scale_log2;       // scale * log2(e)
    const __nv_bfloat16* Q; // [n_seg, seg_rows, 64] (rows read for the extra components)
    __nv_bfloat16* O;       // [n_seg, seg_rows, 64]
    float* lse;             // [n_seg, seg_rows] or null
    ExtraArgs ex;           // ex.on only for SGA (segment = batch*head)
    const float* bias;      // [n_seg, kv_rows] natural-log per-key bias (size-aware variant)
    float inv_scale;        // 1 / scale
    int store32;            // 1: O is 32-byte aligned, rows are stored as four 32-byte sectors
    long long drop_kv;      // failure-detection self-test: the producer never loads this key
                            // tile (global ring index), so its wait expires; -1 in normal use
};

// byte offset of element (row r, column c) in a bias block
__host__ __device__ constexpr uint32_t ext_off(int r, int c) {
    return (uint32_t)((r >> 3) * 256 + (c >> 3) * 128 + (r & 7) * 16 + (c & 7) * 2);
}

// The query tiles of work unit u.  A full unit holds two consecutive tiles of one segment.  When
// a segment has an odd number of tiles its last one is left over, and the left-over tiles of
// segments 2g and 2g + 1 form a mixed unit: each tile of it attends to the keys of its own
// segment, so no unit computes a tile that lies wholly past the end of its segment.  Units come
// in groups of 2 n_pairs + 1: the full units of segment 2g, those of segment 2g + 1, then their
// mixed unit, so that a mixed unit runs while its segments' keys are still in L2.  (With an odd
// segment count the last group has one segment, and its mixed unit repeats that segment as its
// second tile, which is then not stored.)
struct UnitTiles {
    int seg0, seg1;         // segment of query tile 0, 1
    int row0, row1;         // first row of query tile 0, 1 within its segment
    bool mixed;             // tiles of two segments: ring entries (K_0 j, K_1 j), (V_0 j, V_1 j)
    bool dup1;              // tile 1 repeats tile 0 (odd segment count): not stored
};
__device__ __forceinline__ UnitTiles unit_tiles(const TcArgs& p, long long u) {
    UnitTiles x;
    int seg, pair = -1;
    if (p.group == 0) {
        seg = (int)(u / p.n_pairs);
        pair = (int)(u % p.n_pairs);
    } else {
        const int g = (int)(u / p.group), r = (int)(u % p.group);
        const bool last_single = 2 * g + 1 >= p.n_seg;          // the odd segment count's last group
        seg = 2 * g;
        if (r < p.n_pairs) pair = r;
        else if (!last_single && r < 2 * p.n_pairs) { seg = 2 * g + 1; pair = r - p.n_pairs; }
    }
    x.mixed = pair < 0;
    if (!x.mixed) {
        x.seg0 = x.seg1 = seg;
        x.row0 = pair * 2 * BM;
        x.row1 = x.row0 + BM;
        x.dup1 = false;
    } else {
        x.seg0 = seg;
        x.dup1 = seg + 1 >= p.n_seg;
        x.seg1 = x.dup1 ? seg : seg + 1;
        x.row0 = x.row1 = p.last_row0;
    }
    return x;
}
__device__ __forceinline__ bool unit_mixed(const TcArgs& p, long long u) {
    if (p.group == 0) return false;
    const int g = (int)(u / p.group), r = (int)(u % p.group);
    return r == (2 * g + 1 >= p.n_seg ? p.n_pairs : 2 * p.n_pairs);
}

// mbarrier addresses (computed, so that no dynamically indexed array lands in local memory)
struct Bars {
    uint32_t base;
    // Q buffer b holds the two query tiles of the CTA's units with u_local mod 2 == b
    __device__ __forceinline__ uint32_t q_full(uint32_t b) const { return base + 8 * b; }
    __device__ __forceinline__ uint32_t q_empty(uint32_t b) const { return base + 16 + 8 * b; }
    __device__ __forceinline__ uint32_t kv_full(int s) const { return base + 32 + 8 * s; }
    __device__ __forceinline__ uint32_t kv_empty(int s) const { return base + 32 + 8 * (STAGES + s); }
    // S and P of one slot: per buffer, so that no barrier can run two phases ahead of its waiter
    // (a buffer is refilled only after the P it held has been consumed)
    __device__ __forceinline__ uint32_t s_full(uint32_t b) const { return base + 32 + 8 * (2 * STAGES + b); }
    __device__ __forceinline__ uint32_t p_ready(uint32_t b) const { return base + 32 + 8 * (2 * STAGES + 3 + b); }
    __device__ __forceinline__ uint32_t o_done(int t) const { return base + 32 + 8 * (2 * STAGES + 6 + t); }
    __device__ __forceinline__ uint32_t o_free(int t) const { return base + 32 + 8 * (2 * STAGES + 8 + t); }
    __device__ __forceinline__ uint32_t drain() const { return base + 32 + 8 * (2 * STAGES + 10); }
    __device__ __forceinline__ uint32_t q_rot(uint32_t b) const { return base + 32 + 8 * (2 * STAGES + 11 + b); }
    __device__ __forceinline__ uint32_t pv_done(int t) const { return base + 32 + 8 * (2 * STAGES + 13 + t); }
    __device__ __forceinline__ uint32_t turn(int t) const { return base + 32 + 8 * (2 * STAGES + 15 + t); }
};
static_assert(32 + 8 * (2 * STAGES + 17) == NUM_BARS * 8, "barrier block size");

// Key tile processed at step j of a CTA's u_local-th unit.  All CTAs work on units of the same
// head at the same time and sweep its key tiles; consecutive rounds sweep in opposite
// directions, so a round starts on the tiles the previous one touched last (still in L2).  The
// online softmax does not depend on the order.
__device__ __forceinline__ int key_tile(int j, int n_kv, uint32_t u_local) {
    return (u_local & 1) ? n_kv - 1 - j : j;
}

// Bounded wait without the abort check: used only to drain work already in flight.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kTimeoutCycles / 8) {
            atomicExch(&g_status, (int)SGA_ERR_TIMEOUT);
            return;
        }
    }
}

// warp-uniform bounded wait (tcgen05.ld/st that follow are warp-collective)
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    const bool ok = mbar_wait(bar, parity, abort_flag);
    return __all_sync(0xffffffffu, ok);
}

// 32-byte global store (sm_100+), address 32-byte aligned
__device__ __forceinline__ void st_global_v8(void* p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t a4, uint32_t a5, uint32_t a6, uint32_t a7) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 ::"l"(p), "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7) : "memory");
}

__device__ __forceinline__ void ld_row128(uint32_t taddr, float (&s)[128]) {
    uint32_t r[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        tmem_ld32(taddr + 32 * c, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 * c + i] = __uint_as_float(r[i]);
    }
}

// kDefer: run a unit's epilogue after the next unit's first P (for short units; see below)
template <bool kBias, bool kRope, bool kDefer>
__global__ void __launch_bounds__(NUM_THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const TcArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(base);
    const Bars bars{sbase + OFF_BAR};
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (uint32_t b = 0; b < 2; ++b) {
            mbar_init(bars.q_full(b), 1);
            mbar_init(bars.q_empty(b), 2);              // the QKs of the unit's last two slots
            mbar_init(bars.q_rot(b), 256);
        }
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bars.kv_full(s), 1);
            mbar_init(bars.kv_empty(s), 2);
        }
        for (uint32_t b = 0; b < NUM_SBUF; ++b) {
            mbar_init(bars.s_full(b), 1);
            mbar_init(bars.p_ready(b), 128);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bars.o_done(t), 1);
            mbar_init(bars.o_free(t), 128);
            mbar_init(bars.pv_done(t), 1);
            mbar_init(bars.turn(t), 1);
        }
        mbar_init(bars.drain(), 2);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (kBias && warp < 4) {
        // constant ones block for Q (columns 0-1 = 1.0) and zeroed bias blocks; the producer
        // rewrites only columns 0-1 of the bias blocks
        uint32_t* qe = reinterpret_cast<uint32_t*>(base + OFF_QEXT);
        for (int i = threadIdx.x; i < (EXT_BYTES + STAGES * EXT_BYTES) / 4; i += 128) qe[i] = 0u;
        __syncwarp();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        for (int r = threadIdx.x; r < 128; r += 128)
            *reinterpret_cast<uint32_t*>(base + OFF_QEXT + ext_off(r, 0)) = 0x3F803F80u;   // bf16 1.0, 1.0
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int n_kv = p.n_kv_tiles;
    const int last_valid = p.kv_rows - (n_kv - 1) * BN;     // keys in the last tile (1..128)

    if (warp < 4) {
      regs_dec<REGS_CTRL>();                            // warpgroup 0: one instruction for all 4 warps
      if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        // The whole warp runs the loop (warp-uniform state); one elected lane issues.
        uint32_t kv_it = 0, kv_issued = 0, q_issued = 0, u_local = 0;
        bool ok = true;
        for (long long u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++u_local) {
            const UnitTiles ut = unit_tiles(p, u);
            const uint32_t qb = u_local & 1;
            if (!warp_wait(bars.q_empty(qb), ((u_local >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
            if (elect_one()) {
                const uint32_t dst = sbase + OFF_Q + qb * 2 * TILE_BYTES;
                mbar_arrive_expect_tx(bars.q_full(qb), 2 * TILE_BYTES);
                tma_load_3d(dst, &tmQ, bars.q_full(qb), 0, ut.row0, ut.seg0);
                tma_load_3d(dst + TILE_BYTES, &tmQ, bars.q_full(qb), 0, ut.row1, ut.seg1);
            }
            __syncwarp();
            ++q_issued;
            // ring entries: (K j, V j) of the segment (full unit); in a mixed unit (K j of
            // segment 0, K j of segment 1), then (V j of segment 0, V j of segment 1), so that a
            // K entry is released as soon as its two QKs are done (the bias variant has no
            // mixed units)
            const int n_ent = ut.mixed ? 2 * n_kv : n_kv;
            for (int i = 0; i < n_ent; ++i, ++kv_it) {
                const int st = kv_it % STAGES;
                const uint32_t ph = (kv_it / STAGES) & 1;
                const int j = ut.mixed ? (i >> 1) : i;
                const int seg = ut.seg0;
                const int jt = key_tile(j, n_kv, u_local);
                if (!warp_wait(bars.kv_empty(st), ph ^ 1, abort_flag)) { ok = false; break; }
                if (kBias) {
                    // columns 0-1 of key row r: bias/scale as bf16 high + low parts
                    uint8_t* blk = base + OFF_KEXT + st * EXT_BYTES;
                    const float* brow = p.bias + (long long)seg * p.kv_rows + (long long)jt * BN;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = lane * 4 + i;
                        const float b = (jt * BN + r < p.kv_rows) ? __ldg(brow + r) * p.inv_scale : 0.f;
                        const __nv_bfloat16 hi = __float2bfloat16_rn(b);
                        const __nv_bfloat16 lo = __float2bfloat16_rn(b - __bfloat162float(hi));
                        *reinterpret_cast<uint32_t*>(blk + ext_off(r, 0)) =
                            (uint32_t)__bfloat16_as_ushort(hi) | ((uint32_t)__bfloat16_as_ushort(lo) << 16);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                }
                // K and V of one key tile arrive on one barrier; the self-test loads nothing for
                // tile drop_kv, so that barrier never completes
                if ((long long)kv_it != p.drop_kv) {
                    if (elect_one()) {
                        const CUtensorMap* m0 = (ut.mixed && (i & 1)) ? &tmV : &tmK;
                        const CUtensorMap* m1 = ut.mixed ? m0 : &tmV;
                        mbar_arrive_expect_tx(bars.kv_full(st), 2 * TILE_BYTES);
                        tma_load_3d(sbase + OFF_K + st * TILE_BYTES, m0, bars.kv_full(st), 0, jt * BN, seg);
                        tma_load_3d(sbase + OFF_V + st * TILE_BYTES, m1, bars.kv_full(st), 0, jt * BN, ut.seg1);
                    }
                    __syncwarp();
                }
                kv_issued = kv_it + 1;               // entries [0, kv_issued) are issued (but drop_kv)
            }
        }
        if (!ok) {
            // let the copies already issued land before the CTA leaves
            for (uint32_t i = (kv_issued > STAGES ? kv_issued - STAGES : 0); i < kv_issued; ++i)
                if ((long long)i != p.drop_kv) drain_wait(bars.kv_full(i % STAGES), (i / STAGES) & 1);
            for (uint32_t i = (q_issued > 2 ? q_issued - 2 : 0); i < q_issued; ++i)
                drain_wait(bars.q_full(i & 1), (i >> 1) & 1);
        }
      } else if (warp <= 2) {
        // ------------------------------------------------------------------ MMA issuers
        // Slots: the n-th (query tile, key tile) pair of a unit is slot n = 2j + t; the CTA's
        // slots are numbered on across its units (global slot s = u_local * 2 n_kv + n).  Slot s's
        // S goes to buffer s mod 3 and its P is written over it.  Batch G_s (issued by issuer
        // s mod 2 once P(s) is ready) holds PV(s), then QK(s + 3), whose buffer is the one PV(s)
        // has just read; QK(s + 3) may belong to the next unit (its Q tiles sit in the other Q
        // buffer), so the tensor pipe runs on across unit boundaries and every softmax warp finds
        // its next S computed.  The issuers take turns (token through the turn barriers) so the
        // batches reach the tensor pipe in slot order; issuer 0 opens with the first three QKs.
        const int t = warp - 1;
        const uint64_t dQ = smem_desc_sw128(sbase + OFF_Q, 16);
        const uint64_t dK = smem_desc_sw128(sbase + OFF_K, 16);
        const uint64_t dV = smem_desc_sw128(sbase + OFF_V, TILE_BYTES);
        const uint64_t dQe = smem_desc_noswz(sbase + OFF_QEXT, 128, 256);
        const uint64_t dKe = smem_desc_noswz(sbase + OFF_KEXT, 128, 256);
        constexpr uint64_t kTileStep = TILE_BYTES >> 4;
        constexpr uint64_t kExtStep = EXT_BYTES >> 4;
        // in a mixed unit, tile 1's K sits in the V half of the stage and tile 0's V in the K half
        constexpr uint64_t kHalfStep = (uint64_t)(STAGES * TILE_BYTES) >> 4;
        const uint32_t to = tmem + col_o(t);
        const uint32_t n_slots = 2u * (uint32_t)n_kv;
        const uint32_t my_units = (uint32_t)((p.n_units - 1 - blockIdx.x) / gridDim.x + 1);   // grid <= n_units
        const uint32_t total = my_units * n_slots;
        // A position in the CTA's slot sequence: unit ul (the CTA's ul-th), slot n in it, and the
        // unit's first key ring entry (a full unit takes n_kv entries, a mixed one 2 n_kv).
        struct Cursor { uint32_t ul, n, ebase; bool mixed; };
        auto next_unit = [&](Cursor& c) {
            c.n -= n_slots;
            c.ebase += (c.mixed ? 2u : 1u) * (uint32_t)n_kv;
            ++c.ul;
            c.mixed = unit_mixed(p, blockIdx.x + (long long)c.ul * gridDim.x);
        };
        auto cursor_at = [&](uint32_t n0) -> Cursor {
            Cursor c{0u, n0, 0u, unit_mixed(p, blockIdx.x)};
            while (c.n >= n_slots) next_unit(c);
            return c;
        };
        // ring entry read by QK (kv = 0) or PV (kv = 1) of slot c
        auto entry = [&](const Cursor& c, uint32_t kv) -> uint32_t {
            return c.ebase + (c.mixed ? (c.n & ~1u) + kv : c.n >> 1);
        };
        uint32_t turns = 0;
        bool ok = true;
        auto issue_qk = [&](uint32_t s, const Cursor& c) {
            const int st = (int)(entry(c, 0) % STAGES);
            const uint32_t ts = tmem + col_buf(s % NUM_SBUF);
            const uint64_t dq = dQ + (uint64_t)(2 * (c.ul & 1) + (c.n & 1)) * kTileStep;
            const uint64_t dk = dK + (uint64_t)st * kTileStep + ((c.mixed && (c.n & 1)) ? kHalfStep : 0ull);
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk)
                mma_ss(ts, dq + 2 * kk, dk + 2 * kk, IDESC_QK, kk > 0 ? 1u : 0u);
            if (kBias) mma_ss(ts, dQe, dKe + (uint64_t)st * kExtStep, IDESC_QK, 1u);
            mma_commit(bars.s_full(s % NUM_SBUF));
            if (c.n + 2 >= n_slots) mma_commit(bars.q_empty(c.ul & 1));   // the unit's last two QKs
        };
        auto issue_pv = [&](uint32_t s, int st, bool v_low, uint32_t acc) {
            const uint32_t tp = tmem + col_buf(s % NUM_SBUF);
            const uint64_t dv = dV + (uint64_t)st * kTileStep - (v_low ? kHalfStep : 0ull);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
                mma_ts(to, tp + 8 * kk, dv + 128 * kk, IDESC_PV, (acc || kk > 0) ? 1u : 0u);
        };
        auto take_turn = [&]() -> bool {
            const bool got = warp_wait(bars.turn(t), (turns & 1) ^ (t == 0 ? 1u : 0u), abort_flag);
            ++turns;
            return got;
        };
        auto pass_turn = [&]() {
            if (elect_one()) mbar_arrive(bars.turn(t ^ 1));
            __syncwarp();
        };
        if (t == 0) {
            // the first three S: slots 0, 1 (key tile 0) and 2 (key tile 1, or the next unit).
            // Each issuer waits on a unit's Q barrier itself (slots 0-2 alternate issuers).
            Cursor c = cursor_at(0);
            for (uint32_t s = 0; s < 3 && s < total && ok; ++s) {
                const uint32_t e = entry(c, 0);
                if (!warp_wait(bars.kv_full((int)(e % STAGES)), (e / STAGES) & 1, abort_flag) ||
                    !warp_wait(kRope ? bars.q_rot(c.ul & 1) : bars.q_full(c.ul & 1), (c.ul >> 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    issue_qk(s, c);
                    if (c.mixed) mma_commit(bars.kv_empty((int)(e % STAGES)));   // a mixed unit's K entry
                }
                __syncwarp();
                if (++c.n == n_slots) next_unit(c);
            }
        }
        // batch G_s: PV of slot cp, QK of slot cq (three slots on).  Everything the batch waits
        // for is waited for before the turn is taken, so the turn is held only to issue; the one
        // exception is a RoPE unit's rotated Q (see below).
        Cursor cp = cursor_at((uint32_t)t);
        Cursor cq = cursor_at((uint32_t)t + 3);
        for (uint32_t s = (uint32_t)t; s < total && ok; s += 2) {
            const uint32_t j = cp.n >> 1;
            const int st = (int)(entry(cp, 1) % STAGES);
            const bool has_qk = s + 3 < total;
            // with RoPE the next unit's Q is rotated by the softmax warps once they are through
            // this unit's tiles, and one of them may still wait for PV(s): that QK waits for the
            // rotation after PV(s) has been issued
            const bool late_q = kRope && has_qk && cq.n < 3;
            const uint32_t eq = entry(cq, 0);
            if (has_qk) {
                if (!warp_wait(bars.kv_full((int)(eq % STAGES)), (eq / STAGES) & 1, abort_flag)) { ok = false; break; }
                if (!kRope && cq.n < 3 && !warp_wait(bars.q_full(cq.ul & 1), (cq.ul >> 1) & 1, abort_flag)) { ok = false; break; }
            }
            // a mixed unit's V has a ring entry of its own (a full unit's V came with its K)
            if (cp.mixed && !warp_wait(bars.kv_full(st), (entry(cp, 1) / STAGES) & 1, abort_flag)) { ok = false; break; }
            if (!warp_wait(bars.p_ready(s % NUM_SBUF), (s / NUM_SBUF) & 1, abort_flag)) { ok = false; break; }
            if (cp.n < 2 && !warp_wait(bars.o_free(t), (cp.ul & 1) ^ 1, abort_flag)) { ok = false; break; }
            if (!take_turn()) { ok = false; break; }
            tc_fence_after();
            if (elect_one()) {
                issue_pv(s, st, cp.mixed && (cp.n & 1) == 0, j > 0 ? 1u : 0u);
                if (cp.n + 2 >= n_slots) mma_commit(bars.o_done(t));
                if (has_qk && !late_q) issue_qk(s + 3, cq);
            }
            __syncwarp();
            if (late_q) {
                if (!warp_wait(bars.q_rot(cq.ul & 1), (cq.ul >> 1) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                if (elect_one()) issue_qk(s + 3, cq);
                __syncwarp();
            }
            pass_turn();
            if (elect_one()) {
                mma_commit(bars.pv_done(t));
                mma_commit(bars.kv_empty(st));                  // this issuer's last use of the stage
                // a mixed unit's K entry is released by its two QKs
                if (has_qk && cq.mixed) mma_commit(bars.kv_empty((int)(eq % STAGES)));
            }
            __syncwarp();
            cp.n += 2;
            if (cp.n >= n_slots) next_unit(cp);
            cq.n += 2;
            if (cq.n >= n_slots) next_unit(cq);
        }
        // every MMA issued so far completes before TMEM is released
        if (elect_one()) mma_commit(bars.drain());
        __syncwarp();
        drain_wait(bars.drain(), 0);
      }                                                 // warp 3: idle
    } else {
        regs_inc<REGS_SOFTMAX>();
        // ------------------------------------------------------------------ softmax + epilogue
        const int t = (warp - 4) >> 2;                  // query tile of this warpgroup
        const int sub = warp & 3;                       // TMEM lanes [32*sub, 32*sub+32)
        const int r_in_tile = sub * 32 + lane;
        const uint32_t lane_bits = (uint32_t)(sub * 32) << 16;
        const uint32_t tO = tmem + lane_bits + col_o(t);
        const float sl2 = p.scale_log2;
        // RoPE: rotate this thread's row of query tile t of unit uu (the CTA's ul-th) in its Q
        // buffer (128-byte swizzle: the 16-byte chunk c of row r sits at chunk c ^ (r mod 8)), then
        // release it to the MMA.  The first unit's rows are rotated up front, every later unit's
        // as soon as this warpgroup is through the tiles of the unit before it.
        auto rotate_q = [&](long long uu, uint32_t ul) -> bool {
            if (!warp_wait(bars.q_full(ul & 1), (ul >> 1) & 1, abort_flag)) return false;
            const UnitTiles un = unit_tiles(p, uu);
            const int rrow = (t ? un.row1 : un.row0) + r_in_tile;
            if (rrow < p.seg_rows) {
                uint8_t* qrow = base + OFF_Q + (2 * (ul & 1) + t) * TILE_BYTES + r_in_tile * 128;
                float x[64];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 w = *reinterpret_cast<const uint4*>(qrow + ((c ^ (r_in_tile & 7)) * 16));
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) { x[8 * c + 2 * i] = bf16_lo(ww[i]); x[8 * c + 2 * i + 1] = bf16_hi(ww[i]); }
                }
                rope_row64(p.ex.rope, rrow, x);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(qrow + ((c ^ (r_in_tile & 7)) * 16)) =
                        make_uint4(pack_bf16x2(x[8 * c], x[8 * c + 1]), pack_bf16x2(x[8 * c + 2], x[8 * c + 3]),
                                   pack_bf16x2(x[8 * c + 4], x[8 * c + 5]), pack_bf16x2(x[8 * c + 6], x[8 * c + 7]));
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            mbar_arrive(bars.q_rot(ul & 1));
            return true;
        };
        // With kDefer a unit's epilogue runs once this warpgroup has stored the next unit's first
        // P: by then the unit's last PV is long complete.  That matters for short units
        // (frame-local attention, 11 key tiles); for units of whole sequences the host launches
        // the form that runs it straight after the unit, which needs fewer registers.  Either
        // way the row state waits in shared memory.
        float* pend = reinterpret_cast<float*>(base + OFF_PEND) + (threadIdx.x - 128);
        auto epilogue = [&](uint32_t ul) -> bool {
            if (!warp_wait(bars.o_done(t), ul & 1, abort_flag)) return false;
            tc_fence_after();
            float o[64];
            {
                uint32_t r[32];
                tmem_ld32(tO, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]);
                tmem_ld32(tO + 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) o[32 + i] = __uint_as_float(r[i]);
            }
            tc_fence_before();
            mbar_arrive(bars.o_free(t));
            const int seg = __float_as_int(pend[6 * 256]);
            const int row = __float_as_int(pend[7 * 256]);
            if (seg >= 0 && SGA_CHECK_INDEX((long long)seg * p.seg_rows + row, (long long)p.n_seg * p.seg_rows, 10)) {
                const float m = pend[0], l = pend[256];
                if (p.ex.on) {
                    const ExtraRow xr{pend[2 * 256], pend[3 * 256], __float_as_int(pend[4 * 256]), pend[5 * 256]};
                    extra_values<__nv_bfloat16, 64>(p.ex, seg, row, xr, m, 0, o);
                }
                const float inv_l = 1.0f / l;
                const long long grow = (long long)seg * p.seg_rows + row;
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) w[c] = pack_bf16x2(o[2 * c] * inv_l, o[2 * c + 1] * inv_l);
                if (p.store32) {
                    // whole 32-byte sectors: a warp's store writes 32 full sectors, not 32 halves
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        st_global_v8(p.O + grow * 64 + 16 * c, w[8 * c], w[8 * c + 1], w[8 * c + 2], w[8 * c + 3],
                                     w[8 * c + 4], w[8 * c + 5], w[8 * c + 6], w[8 * c + 7]);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(p.O + grow * 64);
#pragma unroll
                    for (int c = 0; c < 8; ++c) dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                }
                if (p.lse) p.lse[grow] = (m + log2f(l)) * 0.69314718055994531f;
            }
            return true;
        };
        uint32_t g_it = 0, u_local = 0, slot_base = 0;
        bool ok = true;
        if (kRope && !rotate_q(blockIdx.x, 0)) ok = false;
        for (long long u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++u_local) {
            const UnitTiles ut = unit_tiles(p, u);
            const int seg = t ? ut.seg1 : ut.seg0;
            const int row = (t ? ut.row1 : ut.row0) + r_in_tile;
            const bool valid = row < p.seg_rows && !(t == 1 && ut.dup1);

            float m = -INFINITY, l = 0.f;
            ExtraRow xr{};
            if (p.ex.on && valid) {
                float q[64];
                load_row64<__nv_bfloat16>(p.Q + ((long long)seg * p.seg_rows + row) * 64, q);
                if (kRope) rope_row64(p.ex.rope, row, q);
                xr = extra_logits<__nv_bfloat16, kRope>(p.ex, seg, row, q, sl2);
                m = fmaxf(xr.s_diag, xr.s_mean);
                if (m != -INFINITY)
                    l = (xr.s_diag == -INFINITY ? 0.f : exp2f(xr.s_diag - m)) +
                        (xr.s_mean == -INFINITY ? 0.f : exp2f(xr.s_mean - m));
            }
            // A row without the extra components has no reference max yet: the unit's first key
            // tile sets it to that tile's row maximum (as a max-first softmax would).
            const bool need_init = __any_sync(0xffffffffu, m == -INFINITY);

            // one key tile of this unit (the first one also sets the reference max where there is
            // none yet, and runs the previous unit's epilogue)
            auto tile = [&](int j, bool first) -> bool {
                // this slot's S, and then its P, live in buffer (global slot) mod 3
                const uint32_t sn = slot_base + 2u * (uint32_t)j + (uint32_t)t;    // global slot
                const uint32_t tS = tmem + lane_bits + col_buf(sn % NUM_SBUF);
                if (!warp_wait(bars.s_full(sn % NUM_SBUF), (sn / NUM_SBUF) & 1, abort_flag)) return false;
                tc_fence_after();
                float s[128];
                ld_row128(tS, s);
                tmem_wait_ld();
                if (key_tile(j, n_kv, u_local) == n_kv - 1 && last_valid < BN) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= last_valid) s[c] = -INFINITY;
                }
                if (first && need_init) {
                    float mx8[8];
#pragma unroll
                    for (int gg = 0; gg < 8; ++gg) {
                        float a = max3f(s[16 * gg], s[16 * gg + 1], s[16 * gg + 2]);
#pragma unroll
                        for (int c = 3; c < 15; c += 2) a = max3f(a, s[16 * gg + c], s[16 * gg + c + 1]);
                        mx8[gg] = fmaxf(a, s[16 * gg + 15]);
                    }
                    const float mx = fmaxf(max3f(mx8[0], mx8[1], mx8[2]),
                                           max3f(max3f(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
                    if (m == -INFINITY) m = mx * sl2;
                }
                // p = 2^(s * scale_log2 - m) against the row's current reference max m (the whole
                // row of S is in registers, so P can go over it at once); the tile sum decides
                // whether that was final
                const uint64_t sc2 = f2_pack(sl2, sl2);
                uint64_t nm2 = f2_pack(-m, -m);
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(s[32 * c + 2 * i], s[32 * c + 2 * i + 1]), sc2, nm2), x0, x1);
                        const float p0 = ex2_approx(x0);
                        const float p1 = ex2_approx(x1);
                        acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16(tS + 16 * c, pk);
                }
                float tsum;
                {
                    float a0, a1;
                    f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
                    tsum = a0 + a1;
                }
                // The reference moves (and O is rescaled) only when a row's logits exceed it by
                // more than 2^kRescaleThreshold.  A tile sum of at most 2^7 puts every p at or
                // below 2^7, so every logit stays at least 1 below that bound: the P just stored
                // is final.  Otherwise (rare) the decision is taken on the row maximum as a
                // max-first softmax takes it, and P is recomputed when the reference moves.
                if (__any_sync(0xffffffffu, !(tsum <= kSumTrigger))) {
                    float mx8[8];
#pragma unroll
                    for (int gg = 0; gg < 8; ++gg) {
                        float a = max3f(s[16 * gg], s[16 * gg + 1], s[16 * gg + 2]);
#pragma unroll
                        for (int c = 3; c < 15; c += 2) a = max3f(a, s[16 * gg + c], s[16 * gg + c + 1]);
                        mx8[gg] = fmaxf(a, s[16 * gg + 15]);
                    }
                    const float mx = fmaxf(max3f(mx8[0], mx8[1], mx8[2]),
                                           max3f(max3f(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
                    const float m_cand = mx * sl2;
                    const bool need = m_cand > m + kRescaleThreshold;
                    if (__any_sync(0xffffffffu, need)) {
                        const float m_new = fmaxf(m, m_cand);
                        const float alpha = ex2_approx(m - m_new);
                        l *= alpha;
                        m = m_new;
                        nm2 = f2_pack(-m, -m);
                        uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
                        tmem_wait_st();
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint32_t pk[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                float x0, x1;
                                f2_unpack(f2_fma(f2_pack(s[32 * c + 2 * i], s[32 * c + 2 * i + 1]), sc2, nm2), x0, x1);
                                const float p0 = ex2_approx(x0);
                                const float p1 = ex2_approx(x1);
                                acc2[i & 3] = f2_add(acc2[i & 3], f2_pack(p0, p1));
                                pk[i] = pack_bf16x2(p0, p1);
                            }
                            tmem_st16(tS + 16 * c, pk);
                        }
                        float a0, a1;
                        f2_unpack(f2_add(f2_add(acc2[0], acc2[1]), f2_add(acc2[2], acc2[3])), a0, a1);
                        tsum = a0 + a1;
                        if (j > 0) {
                            if (!warp_wait(bars.pv_done(t), (g_it - 1) & 1, abort_flag)) return false;
                            tc_fence_after();
                            uint32_t r[32];
#pragma unroll
                            for (int c = 0; c < 2; ++c) {
                                tmem_ld32(tO + 32 * c, r);
                                tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                                tmem_st32(tO + 32 * c, r);
                            }
                        }
                    }
                }
                l += tsum;
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bars.p_ready(sn % NUM_SBUF));
                // the previous unit's epilogue, now that this unit's first P is out
                if (kDefer && first && u_local > 0 && !epilogue(u_local - 1)) return false;
                return true;
            };
            if (!tile(0, true)) { ok = false; break; }
            ++g_it;
            for (int j = 1; j < n_kv; ++j, ++g_it)
                if (!tile(j, false)) { ok = false; break; }
            if (!ok) break;
            slot_base += 2u * (uint32_t)n_kv;
            if (kRope && u + gridDim.x < p.n_units && !rotate_q(u + gridDim.x, u_local + 1)) { ok = false; break; }
            pend[0] = m;
            pend[256] = l;
            pend[2 * 256] = xr.s_diag;
            pend[3 * 256] = xr.s_mean;
            pend[4 * 256] = __int_as_float(xr.loo);
            pend[5 * 256] = xr.inv_c;
            pend[6 * 256] = __int_as_float(valid ? seg : -1);
            pend[7 * 256] = __int_as_float(row);
            if (!kDefer && !epilogue(u_local)) { ok = false; break; }
        }
        if (kDefer && ok && u_local > 0) epilogue(u_local - 1);
    }

    // ---------------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace tc
}  // namespace sga
