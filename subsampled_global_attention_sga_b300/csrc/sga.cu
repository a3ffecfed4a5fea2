// sga.cu -- libsga: the C ABI declared in include/sga.h, the host-side plan builder and the
// kernel launchers.  Single translation unit: every kernel of the library is included here.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "attn_simt.cuh"
#include "attn_tc.cuh"
#include "compact.cuh"
#include "compact_rope.cuh"
#include "compact_noalloc.cuh"
#include "merge.cuh"
#include "rope.cuh"

namespace {

constexpr uint32_t kPlanMagic = 0x53474150u;   // "SGAP"
constexpr int kCompactRowsPerChunk = 2048;
// bf16 with the rotation: work items of the persistent TMA-fed kernel (2 CTAs per SM), short
// enough that the items spread evenly over the CTAs (a multiple of its 64-row stage)
constexpr int kCompactRowsPerChunkRope = 1024;
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool init = false;
    int sm_count = 0;
    bool tc_ready[2][2][2] = {};                               // attn_tc_kernel<bias, rope, defer> ready
    size_t cr_smem = 0;                                        // compact_rope_kernel: smem enabled
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

}  // namespace

struct sga_plan_s {
    uint32_t magic;
    sga_config cfg;
    int device;
    long long L, T, S, D;
    int rows_per_chunk;     // compaction rows per block (work item of the RoPE kernel)
    int n_chunks;
    int32_t* d_slot;        // [T], padded with -1 to a multiple of 64 entries (whole 256-byte copies)
    int32_t* d_kv_index;    // [S]
    int32_t* d_frame_off;   // [N+1]
    float* d_partials;      // [B*H, n_chunks, 128]
    float2* d_rope;         // [rope_P, 16] (cos, sin), or null without the rotary embedding
    int rope_P;
    std::vector<int32_t> h_kv_index;
    std::vector<int32_t> h_frame_off;
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

sga_status device_info(int dev, DeviceInfo** out) {
    if (dev < 0 || dev >= kMaxDevices) return SGA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.init) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SGA_ERR_CUDA;
        d.init = true;
    }
    *out = &d;
    return SGA_OK;
}

sga_status current_device(int* dev) {
    return cudaGetDevice(dev) == cudaSuccess ? SGA_OK : SGA_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D map over a contiguous [n_seg, rows, 64] bf16 tensor, box = 128 rows x 64 columns,
// 128-byte swizzle (rows are exactly 128 bytes), zero fill outside [0, rows).
sga_status make_map(CUtensorMap* map, const void* ptr, long long rows, long long n_seg, int box_rows = 128) {
    auto fn = encode_fn();
    if (!fn) return SGA_ERR_CUDA;
    if (rows <= 0 || n_seg <= 0 || rows > 0x7FFFFFFFLL || n_seg > 0x7FFFFFFFLL) return SGA_ERR_UNSUPPORTED;
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)n_seg};
    cuuint64_t strides[2] = {64 * 2, (cuuint64_t)rows * 64 * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SGA_OK : SGA_ERR_CUDA;
}

sga_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? SGA_OK : SGA_ERR_CUDA;
}

// Problem description shared by the three attention entry points.
struct AttnProblem {
    int dtype;
    int kernel;
    int n_seg;
    long long seg_rows;
    long long kv_rows;
    const void* Q;
    const void* Kt;
    const void* Vt;
    void* O;
    float* lse;
    float scale;
    sga::ExtraArgs ex;
    const float* bias;      // per-key natural-log bias [n_seg, kv_rows], or null
    bool rope;              // rotate Q (and the extras' keys) with ex.rope
    long long drop_kv;      // failure-detection self-test only (-1: off)
};

// The tensor-core kernel instantiation for a bias setting, checked once per device: its
// setmaxnreg split assumes exactly LAUNCH_REGS registers per thread at launch (any other count
// would leave setmaxnreg.inc unsatisfiable), and it needs the large dynamic shared memory.
template <bool kBias, bool kRope, bool kDefer>
sga_status prepare_tc(DeviceInfo* di) {
    namespace T = sga::tc;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (di->tc_ready[kBias][kRope][kDefer]) return SGA_OK;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, T::attn_tc_kernel<kBias, kRope, kDefer>) != cudaSuccess) return SGA_ERR_CUDA;
    if (fa.numRegs != (int)T::LAUNCH_REGS) return SGA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(T::attn_tc_kernel<kBias, kRope, kDefer>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             T::SMEM_BYTES) != cudaSuccess)
        return SGA_ERR_CUDA;
    di->tc_ready[kBias][kRope][kDefer] = true;
    return SGA_OK;
}

// Launch one instantiation of the tensor-core kernel.
template <bool kBias, bool kRope, bool kDefer>
sga_status launch_tc(DeviceInfo* di, long long grid, const CUtensorMap& mq, const CUtensorMap& mk,
                     const CUtensorMap& mv, const sga::tc::TcArgs& a, cudaStream_t stream) {
    namespace T = sga::tc;
    sga_status st = prepare_tc<kBias, kRope, kDefer>(di);
    if (st != SGA_OK) return st;
    T::attn_tc_kernel<kBias, kRope, kDefer><<<(unsigned)grid, T::NUM_THREADS, T::SMEM_BYTES, stream>>>(mq, mk, mv, a);
    return launch_status();
}

sga_status run_attention(const AttnProblem& pb, cudaStream_t stream) {
    int dev;
    if (current_device(&dev) != SGA_OK) return SGA_ERR_CUDA;
    DeviceInfo* di;
    sga_status st = device_info(dev, &di);
    if (st != SGA_OK) return st;
    const float scale_log2 = pb.scale * 1.4426950408889634f;
    int kern = pb.kernel;
    if (kern == SGA_KERNEL_AUTO) kern = (pb.dtype == SGA_BF16) ? SGA_KERNEL_TC : SGA_KERNEL_SIMT;
    if (kern == SGA_KERNEL_TC) {
        if (pb.dtype != SGA_BF16) return SGA_ERR_UNSUPPORTED;
        if (pb.seg_rows > 0x7FFFFFFFLL || pb.kv_rows > 0x7FFFFFFFLL) return SGA_ERR_UNSUPPORTED;
        namespace T = sga::tc;
        if (pb.bias && pb.rope) return SGA_ERR_UNSUPPORTED;
        CUtensorMap mq, mk, mv;
        if ((st = make_map(&mq, pb.Q, pb.seg_rows, pb.n_seg)) != SGA_OK) return st;
        if ((st = make_map(&mk, pb.Kt, pb.kv_rows, pb.n_seg)) != SGA_OK) return st;
        if ((st = make_map(&mv, pb.Vt, pb.kv_rows, pb.n_seg)) != SGA_OK) return st;
        T::TcArgs a;
        a.n_seg = pb.n_seg;
        a.seg_rows = (int)pb.seg_rows;
        a.kv_rows = (int)pb.kv_rows;
        const long long q_tiles = (pb.seg_rows + T::BM - 1) / T::BM;
        // a segment's left-over query tile (odd tile count) goes into a mixed unit with the next
        // segment's; the bias variant keeps it in a unit of its own (its second tile unused)
        const bool mixed = (q_tiles & 1) && !pb.bias;
        a.n_pairs = (int)(mixed ? q_tiles / 2 : (q_tiles + 1) / 2);
        a.n_kv_tiles = (int)((pb.kv_rows + T::BN - 1) / T::BN);
        a.n_units = (long long)a.n_seg * a.n_pairs + (mixed ? (a.n_seg + 1) / 2 : 0);
        a.group = mixed ? 2 * a.n_pairs + 1 : 0;
        a.last_row0 = (int)((q_tiles - 1) * T::BM);
        a.scale_log2 = scale_log2;
        a.Q = reinterpret_cast<const __nv_bfloat16*>(pb.Q);
        a.O = reinterpret_cast<__nv_bfloat16*>(pb.O);
        a.lse = pb.lse;
        a.ex = pb.ex;
        a.bias = pb.bias;
        a.inv_scale = 1.0f / pb.scale;
        a.drop_kv = pb.drop_kv;
        // outputs are only required to be 16-byte aligned; whole-sector stores need 32
        a.store32 = (reinterpret_cast<uintptr_t>(pb.O) & 31) == 0 ? 1 : 0;
        const long long grid = a.n_units < di->sm_count ? a.n_units : di->sm_count;
        // short units (up to 32 key tiles: frame-local attention, small layers) defer each unit's
        // epilogue past the next unit's first P; units of whole sequences do not need to
        const bool defer = a.n_kv_tiles <= 32;
        if (pb.bias)
            return defer ? launch_tc<true, false, true>(di, grid, mq, mk, mv, a, stream)
                         : launch_tc<true, false, false>(di, grid, mq, mk, mv, a, stream);
        if (pb.rope)
            return defer ? launch_tc<false, true, true>(di, grid, mq, mk, mv, a, stream)
                         : launch_tc<false, true, false>(di, grid, mq, mk, mv, a, stream);
        return defer ? launch_tc<false, false, true>(di, grid, mq, mk, mv, a, stream)
                     : launch_tc<false, false, false>(di, grid, mq, mk, mv, a, stream);
    }
    if (kern != SGA_KERNEL_SIMT) return SGA_ERR_INVALID_ARG;
    sga::SimtArgs a;
    a.seg_rows = pb.seg_rows;
    a.kv_rows = pb.kv_rows;
    a.Q = pb.Q;
    a.Kt = pb.Kt;
    a.Vt = pb.Vt;
    a.O = pb.O;
    a.lse = pb.lse;
    a.scale_log2 = scale_log2;
    a.ex = pb.ex;
    a.bias = pb.bias;
    const long long gx = (pb.seg_rows + sga::kSimtRows - 1) / sga::kSimtRows;
    if (gx > 0x7FFFFFFFLL || pb.n_seg > 65535) return SGA_ERR_UNSUPPORTED;
    dim3 grid((unsigned)gx, (unsigned)pb.n_seg);
    if (pb.dtype == SGA_BF16)
        sga::attn_simt_kernel<__nv_bfloat16><<<grid, sga::kSimtRows, 0, stream>>>(a);
    else if (pb.dtype == SGA_F32)
        sga::attn_simt_kernel<float><<<grid, sga::kSimtRows, 0, stream>>>(a);
    else
        return SGA_ERR_UNSUPPORTED;
    return launch_status();
}

sga::RopeArgs rope_args(sga_plan_t plan) {
    sga::RopeArgs r;
    std::memset(&r, 0, sizeof(r));
    if (plan->cfg.rope) {
        r.on = 1;
        r.tab = plan->d_rope;
        r.P = plan->rope_P;
        r.L = (int)plan->L;
        r.n_special = plan->cfg.n_special;
        r.grid_w = plan->cfg.grid_w;
        r.pos_offset = plan->cfg.rope_pos_offset;
    }
    return r;
}

sga_status check_plan(sga_plan_t plan) {
    if (!plan || plan->magic != kPlanMagic) return SGA_ERR_PLAN_MISMATCH;
    int dev;
    if (current_device(&dev) != SGA_OK) return SGA_ERR_CUDA;
    return dev == plan->device ? SGA_OK : SGA_ERR_PLAN_MISMATCH;
}

sga_status check_common(int dtype, int head_dim, int kernel) {
    if (head_dim != 64) return SGA_ERR_UNSUPPORTED;
    if (dtype != SGA_BF16 && dtype != SGA_F32) return SGA_ERR_UNSUPPORTED;
    if (kernel < SGA_KERNEL_AUTO || kernel > SGA_KERNEL_SIMT) return SGA_ERR_INVALID_ARG;
    if (kernel == SGA_KERNEL_TC && dtype != SGA_BF16) return SGA_ERR_UNSUPPORTED;
    return SGA_OK;
}

// Kept set S of a layer.  Membership of a frame's slots depends only on the frame's phase
// (and on frame 0 being the dense reference), so one mask per phase is built and reused.
//   kept: frame 0 when it is the dense reference; the n_special camera/register slots of every
//   frame; a patch (r, c) with r = phi_r (mod s_h) and c = phi_c (mod s_w), the first patch of
//   its window, where phi = 0 without the phase shift and phi_r = (f div s_w) mod s_h,
//   phi_c = f mod s_w with it.
void build_plan(const sga_config& c, std::vector<int32_t>& slot, std::vector<int32_t>& kv,
                std::vector<int32_t>& off) {
    const long long L = (long long)c.n_special + (long long)c.grid_h * c.grid_w;
    const long long T = L * c.N;
    slot.assign((size_t)T, -1);
    kv.clear();
    kv.reserve((size_t)T);
    off.assign((size_t)c.N + 1, 0);
    std::vector<uint8_t> mask((size_t)L);
    int cached_pr = -1, cached_pc = -1;
    for (int f = 0; f < c.N; ++f) {
        off[f] = (int32_t)kv.size();
        const bool dense = (f == 0 && c.ref_frame_dense) || (c.s_h == 1 && c.s_w == 1);
        const int pr = c.phase_shift ? (f / c.s_w) % c.s_h : 0;
        const int pc = c.phase_shift ? f % c.s_w : 0;
        if (!dense && (pr != cached_pr || pc != cached_pc)) {
            for (long long p = 0; p < L; ++p) {
                if (p < c.n_special) { mask[p] = 1; continue; }
                const long long r = (p - c.n_special) / c.grid_w, col = (p - c.n_special) % c.grid_w;
                mask[p] = (r >= pr && (r - pr) % c.s_h == 0 && col >= pc && (col - pc) % c.s_w == 0) ? 1 : 0;
            }
            cached_pr = pr;
            cached_pc = pc;
        }
        for (long long p = 0; p < L; ++p) {
            const long long t = (long long)f * L + p;
            if (dense || mask[p]) {
                slot[t] = (int32_t)kv.size();
                kv.push_back((int32_t)t);
            }
        }
    }
    off[c.N] = (int32_t)kv.size();
}

sga_status check_config(const sga_config* cfg) {
    if (!cfg) return SGA_ERR_INVALID_ARG;
    const sga_config& c = *cfg;
    if (c.B <= 0 || c.H <= 0 || c.N <= 0 || c.grid_h <= 0 || c.grid_w <= 0 || c.n_special < 0 ||
        c.s_h <= 0 || c.s_w <= 0)
        return SGA_ERR_INVALID_ARG;
    if (c.mean_mode != SGA_MEAN_LOO && c.mean_mode != SGA_MEAN_GLOBAL) return SGA_ERR_INVALID_ARG;
    if (c.rope != 0 && c.rope != 1) return SGA_ERR_INVALID_ARG;
    if (c.rope && (!(c.rope_base > 1.0f) || !std::isfinite(c.rope_base) || c.rope_pos_offset < 0 ||
                   (long long)c.rope_pos_offset + (c.grid_h > c.grid_w ? c.grid_h : c.grid_w) > 4096))
        return SGA_ERR_INVALID_ARG;
    sga_status st = check_common(c.dtype, c.head_dim, c.kernel);
    if (st != SGA_OK) return st;
    const long long L = (long long)c.n_special + (long long)c.grid_h * c.grid_w;
    if (L * c.N > 0x7FFFFFFFLL || (long long)c.B * c.H > 0x7FFFFFFFLL) return SGA_ERR_UNSUPPORTED;
    return SGA_OK;
}

}  // namespace

extern "C" {

const char* sga_status_string(sga_status s) {
    switch (s) {
        case SGA_OK: return "ok";
        case SGA_ERR_INVALID_ARG: return "invalid argument";
        case SGA_ERR_UNSUPPORTED: return "unsupported (head_dim must be 64; dtype bf16 or f32)";
        case SGA_ERR_ALIGNMENT: return "tensor pointer not 16-byte aligned";
        case SGA_ERR_CUDA: return "CUDA runtime or driver error";
        case SGA_ERR_TIMEOUT: return "kernel wait timed out";
        case SGA_ERR_PLAN_MISMATCH: return "plan invalid or created for another device";
        case SGA_ERR_SCRATCH_LIMIT: return "problem exceeds the fixed scratch of sga_compact_noalloc";
        case SGA_ERR_DEBUG_CHECK: return "a kernel's index check failed (debug build; see sga_debug_report)";
    }
    return "unknown status";
}

#ifndef SGA_SOURCE_HASH
#define SGA_SOURCE_HASH "unknown"
#endif
#ifdef SGA_DEBUG
#define SGA_BUILD_KIND "debug (index checks) "
#else
#define SGA_BUILD_KIND ""
#endif
const char* sga_build_info(void) {
    return "libsga sm_103a (tcgen05/TMEM/TMA attention, CUDA-core fp32 path) v2 " SGA_BUILD_KIND "src=" SGA_SOURCE_HASH;
}

sga_status sga_debug_report(int64_t* site, int64_t* index, int64_t* bound, int64_t* count) {
#ifdef SGA_DEBUG
    if (cudaDeviceSynchronize() != cudaSuccess) return SGA_ERR_CUDA;
    unsigned long long w[4] = {0, 0, 0, 0};
    if (cudaMemcpyFromSymbol(w, sga::g_debug_word, sizeof(w)) != cudaSuccess) return SGA_ERR_CUDA;
    const unsigned long long zero[4] = {0, 0, 0, 0};
    if (cudaMemcpyToSymbol(sga::g_debug_word, zero, sizeof(zero)) != cudaSuccess) return SGA_ERR_CUDA;
    if (site) *site = (int64_t)w[0];
    if (index) *index = (int64_t)w[1];
    if (bound) *bound = (int64_t)w[2];
    if (count) *count = (int64_t)w[3];
    return SGA_OK;
#else
    (void)site; (void)index; (void)bound; (void)count;
    return SGA_ERR_UNSUPPORTED;
#endif
}

}  // extern "C"

namespace {

// Upload a kept set (slot map, ascending kept list, frame offsets) as a plan on `device`.
sga_status upload_plan(const sga_config& c, const std::vector<int32_t>& slot, const std::vector<int32_t>& kv,
                       const std::vector<int32_t>& off, int device, sga_plan_t* out) {
    const long long L = (long long)c.n_special + (long long)c.grid_h * c.grid_w;
    const long long T = L * c.N;
    sga_plan_s* plan = new (std::nothrow) sga_plan_s();
    if (!plan) return SGA_ERR_CUDA;
    plan->magic = kPlanMagic;
    plan->cfg = c;
    plan->device = device;
    plan->L = L;
    plan->T = T;
    plan->S = (long long)kv.size();
    plan->D = T - plan->S;
    plan->rows_per_chunk = (c.rope && c.dtype == SGA_BF16) ? kCompactRowsPerChunkRope : kCompactRowsPerChunk;
    plan->n_chunks = (int)((T + plan->rows_per_chunk - 1) / plan->rows_per_chunk);
    plan->h_kv_index = kv;
    plan->h_frame_off = off;
    plan->d_slot = nullptr;
    plan->d_kv_index = nullptr;
    plan->d_frame_off = nullptr;
    plan->d_partials = nullptr;
    plan->d_rope = nullptr;
    plan->rope_P = 0;
    std::vector<float> rope_tab;
    if (c.rope) {
        // positions 0 .. max(grid) - 1 + offset; angle pos * base^(-j/16), computed in double
        plan->rope_P = (c.grid_h > c.grid_w ? c.grid_h : c.grid_w) + c.rope_pos_offset;
        rope_tab.resize((size_t)plan->rope_P * 32);
        for (int pos = 0; pos < plan->rope_P; ++pos)
            for (int j = 0; j < 16; ++j) {
                const double ang = pos * std::pow((double)c.rope_base, -2.0 * j / 32.0);
                rope_tab[(size_t)(pos * 16 + j) * 2] = (float)std::cos(ang);
                rope_tab[(size_t)(pos * 16 + j) * 2 + 1] = (float)std::sin(ang);
            }
    }

    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) {
        delete plan;
        return SGA_ERR_CUDA;
    }
    bool okc = true;
    const size_t part_bytes = (size_t)c.B * c.H * plan->n_chunks * 128 * sizeof(float);
    const size_t slot_n = (size_t)((T + 63) / 64) * 64;
    okc = okc && cudaMalloc(&plan->d_slot, sizeof(int32_t) * slot_n) == cudaSuccess;
    okc = okc && cudaMemset(plan->d_slot, 0xFF, sizeof(int32_t) * slot_n) == cudaSuccess;
    okc = okc && cudaMalloc(&plan->d_kv_index, sizeof(int32_t) * (size_t)(plan->S > 0 ? plan->S : 1)) == cudaSuccess;
    okc = okc && cudaMalloc(&plan->d_frame_off, sizeof(int32_t) * (size_t)(c.N + 1)) == cudaSuccess;
    okc = okc && cudaMalloc(&plan->d_partials, part_bytes) == cudaSuccess;
    if (c.rope) {
        okc = okc && cudaMalloc(&plan->d_rope, sizeof(float) * rope_tab.size()) == cudaSuccess;
        okc = okc && cudaMemcpy(plan->d_rope, rope_tab.data(), sizeof(float) * rope_tab.size(),
                                cudaMemcpyHostToDevice) == cudaSuccess;
    }
    okc = okc && cudaMemcpy(plan->d_slot, slot.data(), sizeof(int32_t) * (size_t)T, cudaMemcpyHostToDevice) == cudaSuccess;
    if (plan->S > 0)
        okc = okc && cudaMemcpy(plan->d_kv_index, kv.data(), sizeof(int32_t) * (size_t)plan->S,
                                cudaMemcpyHostToDevice) == cudaSuccess;
    okc = okc && cudaMemcpy(plan->d_frame_off, off.data(), sizeof(int32_t) * (size_t)(c.N + 1),
                            cudaMemcpyHostToDevice) == cudaSuccess;
    okc = okc && cudaDeviceSynchronize() == cudaSuccess;
    DeviceInfo* di;
    okc = okc && device_info(device, &di) == SGA_OK;
    cudaSetDevice(prev);
    if (!okc) {
        sga_plan_destroy(plan);
        return SGA_ERR_CUDA;
    }
    *out = plan;
    return SGA_OK;
}

// Generalised kept set ("RegimeVGGT ..." Key design 3): rational per-axis window sizes
// sigma = num/den >= 1, a window keeping its first position ceil(i*sigma); with the phase
// shift the positions move by phi_r = (f div t_w) mod t_h, phi_c = f mod t_w with the integer
// tiles t = ceil(sigma); frame 0 (when dense) and the camera/register tokens kept; protected
// tokens kept in full.  Exact integer arithmetic.
bool window_start(long long x, long long phi, long long num, long long den) {
    if (x < phi) return false;
    const long long y = x - phi;
    if (y == 0) return true;
    const long long i = ((y - 1) * den) / num + 1;     // first window whose start is >= y
    return (i * num + den - 1) / den == y;
}

sga_status build_plan_general(const sga_grid_spec& g, const int32_t* prot, int64_t n_prot,
                              std::vector<int32_t>& slot, std::vector<int32_t>& kv, std::vector<int32_t>& off) {
    const long long L = (long long)g.n_special + (long long)g.grid_h * g.grid_w;
    const long long T = L * g.N;
    std::vector<uint8_t> kept((size_t)T, 0);
    for (int64_t i = 0; i < n_prot; ++i) {
        if (prot[i] < 0 || prot[i] >= T) return SGA_ERR_INVALID_ARG;
        kept[(size_t)prot[i]] = 1;
    }
    const long long th = (g.sh_num + g.sh_den - 1) / g.sh_den, tw = (g.sw_num + g.sw_den - 1) / g.sw_den;
    std::vector<uint8_t> row_ok((size_t)g.grid_h), col_ok((size_t)g.grid_w);
    slot.assign((size_t)T, -1);
    kv.clear();
    off.assign((size_t)g.N + 1, 0);
    for (int f = 0; f < g.N; ++f) {
        off[f] = (int32_t)kv.size();
        const long long pr = g.phase_shift ? (f / tw) % th : 0;
        const long long pc = g.phase_shift ? f % tw : 0;
        for (int r = 0; r < g.grid_h; ++r) row_ok[r] = window_start(r, pr, g.sh_num, g.sh_den);
        for (int c = 0; c < g.grid_w; ++c) col_ok[c] = window_start(c, pc, g.sw_num, g.sw_den);
        const bool dense = f == 0 && g.ref_frame_dense;
        for (long long p = 0; p < L; ++p) {
            const long long t = (long long)f * L + p;
            bool keep = dense || p < g.n_special || kept[(size_t)t];
            if (!keep) {
                const long long q = p - g.n_special;
                keep = row_ok[q / g.grid_w] && col_ok[q % g.grid_w];
            }
            if (keep) {
                slot[(size_t)t] = (int32_t)kv.size();
                kv.push_back((int32_t)t);
            }
        }
    }
    off[g.N] = (int32_t)kv.size();
    return SGA_OK;
}

sga_status check_grid_spec(const sga_grid_spec* g) {
    if (!g) return SGA_ERR_INVALID_ARG;
    if (g->N <= 0 || g->grid_h <= 0 || g->grid_w <= 0 || g->n_special < 0 || g->sh_den <= 0 || g->sw_den <= 0 ||
        g->sh_num < g->sh_den || g->sw_num < g->sw_den)
        return SGA_ERR_INVALID_ARG;
    const long long L = (long long)g->n_special + (long long)g->grid_h * g->grid_w;
    if (L * g->N > 0x7FFFFFFFLL) return SGA_ERR_UNSUPPORTED;
    return SGA_OK;
}

}  // namespace

extern "C" {

sga_status sga_plan_create(const sga_config* cfg, int device, sga_plan_t* out) {
    if (!cfg || !out) return SGA_ERR_INVALID_ARG;
    *out = nullptr;
    sga_status st = check_config(cfg);
    if (st != SGA_OK) return st;
    std::vector<int32_t> slot, kv, off;
    build_plan(*cfg, slot, kv, off);
    return upload_plan(*cfg, slot, kv, off, device, out);
}

sga_status sga_plan_create_from_index(const sga_config* cfg, const int32_t* kv_index, int64_t S, int device,
                                      sga_plan_t* out) {
    if (!cfg || !out || (S > 0 && !kv_index) || S < 0) return SGA_ERR_INVALID_ARG;
    *out = nullptr;
    sga_status st = check_config(cfg);
    if (st != SGA_OK) return st;
    const sga_config& c = *cfg;
    const long long L = (long long)c.n_special + (long long)c.grid_h * c.grid_w;
    const long long T = L * c.N;
    if (S > T) return SGA_ERR_INVALID_ARG;
    std::vector<int32_t> slot((size_t)T, -1), kv(kv_index, kv_index + S), off((size_t)c.N + 1, 0);
    for (int64_t i = 0; i < S; ++i) {
        if (kv[i] < 0 || kv[i] >= T || (i > 0 && kv[i] <= kv[i - 1])) return SGA_ERR_INVALID_ARG;
        slot[(size_t)kv[i]] = (int32_t)i;
    }
    // off[f] = number of kept tokens before frame f
    int64_t i = 0;
    for (int f = 0; f <= c.N; ++f) {
        while (i < S && kv[i] < (long long)f * L) ++i;
        off[f] = (int32_t)i;
    }
    return upload_plan(c, slot, kv, off, device, out);
}

sga_status sga_plan_host_general(const sga_grid_spec* spec, const int32_t* protected_tokens, int64_t n_protected,
                                 int32_t* kv_index, int32_t* frame_off, int32_t* slot, int64_t* S_out) {
    if (!kv_index || !frame_off || !S_out || n_protected < 0 || (n_protected > 0 && !protected_tokens))
        return SGA_ERR_INVALID_ARG;
    sga_status st = check_grid_spec(spec);
    if (st != SGA_OK) return st;
    std::vector<int32_t> sl, kv, off;
    if ((st = build_plan_general(*spec, protected_tokens, n_protected, sl, kv, off)) != SGA_OK) return st;
    std::memcpy(kv_index, kv.data(), sizeof(int32_t) * kv.size());
    std::memcpy(frame_off, off.data(), sizeof(int32_t) * off.size());
    if (slot) std::memcpy(slot, sl.data(), sizeof(int32_t) * sl.size());
    *S_out = (int64_t)kv.size();
    return SGA_OK;
}

sga_status sga_plan_host(const sga_config* cfg, int32_t* kv_index, int32_t* frame_off,
                         int32_t* slot, int64_t* S_out) {
    if (!kv_index || !frame_off || !S_out) return SGA_ERR_INVALID_ARG;
    sga_status st = check_config(cfg);
    if (st != SGA_OK) return st;
    std::vector<int32_t> sl, kv, off;
    build_plan(*cfg, sl, kv, off);
    std::memcpy(kv_index, kv.data(), sizeof(int32_t) * kv.size());
    std::memcpy(frame_off, off.data(), sizeof(int32_t) * off.size());
    if (slot) std::memcpy(slot, sl.data(), sizeof(int32_t) * sl.size());
    *S_out = (int64_t)kv.size();
    return SGA_OK;
}

sga_status sga_plan_info(sga_plan_t plan, int64_t* T, int64_t* S, int64_t* dropped) {
    if (!plan || plan->magic != kPlanMagic) return SGA_ERR_PLAN_MISMATCH;
    if (T) *T = plan->T;
    if (S) *S = plan->S;
    if (dropped) *dropped = plan->D;
    return SGA_OK;
}

sga_status sga_plan_copy_indices(sga_plan_t plan, int32_t* kv_index, int32_t* frame_off) {
    if (!plan || plan->magic != kPlanMagic) return SGA_ERR_PLAN_MISMATCH;
    if (kv_index && plan->S > 0) std::memcpy(kv_index, plan->h_kv_index.data(), sizeof(int32_t) * (size_t)plan->S);
    if (frame_off) std::memcpy(frame_off, plan->h_frame_off.data(), sizeof(int32_t) * (size_t)(plan->cfg.N + 1));
    return SGA_OK;
}

void sga_plan_destroy(sga_plan_t plan) {
    if (!plan || plan->magic != kPlanMagic) return;
    int prev = -1;
    const bool switched = cudaGetDevice(&prev) == cudaSuccess && cudaSetDevice(plan->device) == cudaSuccess;
    if (switched) cudaDeviceSynchronize();
    cudaFree(plan->d_slot);
    cudaFree(plan->d_kv_index);
    cudaFree(plan->d_frame_off);
    cudaFree(plan->d_partials);
    cudaFree(plan->d_rope);
    if (switched) cudaSetDevice(prev);
    plan->magic = 0;
    delete plan;
}

sga_status sga_compact(sga_plan_t plan, const void* K, const void* V, void* K_S, void* V_S,
                       float* k_sum, float* v_sum, void* stream) {
    sga_status st = check_plan(plan);
    if (st != SGA_OK) return st;
    if (!K || !V || !K_S || !V_S || !k_sum || !v_sum) return SGA_ERR_INVALID_ARG;
    if (!aligned16(K) || !aligned16(V) || !aligned16(K_S) || !aligned16(V_S) || !aligned16(k_sum) ||
        !aligned16(v_sum))
        return SGA_ERR_ALIGNMENT;
    const sga_config& c = plan->cfg;
    const int BH = c.B * c.H;
    if (BH > 65535) return SGA_ERR_UNSUPPORTED;
    sga::CompactArgs a;
    a.T = plan->T;
    a.S = plan->S;
    a.rows_per_chunk = plan->rows_per_chunk;
    a.n_chunks = plan->n_chunks;
    a.slot = plan->d_slot;
    a.K = K;
    a.V = V;
    a.KS = K_S;
    a.VS = V_S;
    a.partials = plan->d_partials;
    a.rope = rope_args(plan);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    dim3 grid((unsigned)plan->n_chunks, (unsigned)BH);
    const size_t rope_smem = c.rope ? sizeof(float2) * (size_t)plan->rope_P * sga::kRopeTabStride : 0;
    if (c.dtype == SGA_BF16) {
        if (c.rope) {
            // persistent TMA-fed kernel: the rotation needs the loads decoupled from the compute
            namespace R = sga::cr;
            int dev;
            DeviceInfo* di;
            if (current_device(&dev) != SGA_OK) return SGA_ERR_CUDA;
            if ((st = device_info(dev, &di)) != SGA_OK) return st;
            const size_t smem = R::smem_bytes(plan->rope_P);
            if (smem > 227 * 1024) return SGA_ERR_UNSUPPORTED;
            {
                std::lock_guard<std::mutex> lk(g_dev_mu);
                if (di->cr_smem < smem) {
                    if (cudaFuncSetAttribute(R::compact_rope_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem) != cudaSuccess)
                        return SGA_ERR_CUDA;
                    di->cr_smem = smem;
                }
            }
            CUtensorMap mk, mv;
            if ((st = make_map(&mk, K, plan->T, BH, R::kStageRows)) != SGA_OK) return st;
            if ((st = make_map(&mv, V, plan->T, BH, R::kStageRows)) != SGA_OK) return st;
            R::Args ra;
            ra.T = plan->T;
            ra.S = plan->S;
            ra.rows_per_chunk = plan->rows_per_chunk;
            ra.n_chunks = plan->n_chunks;
            ra.n_items = (long long)BH * plan->n_chunks;
            ra.KS = reinterpret_cast<__nv_bfloat16*>(K_S);
            ra.VS = reinterpret_cast<__nv_bfloat16*>(V_S);
            ra.partials = plan->d_partials;
            ra.rope = a.rope;
            ra.slot = plan->d_slot;
            const long long cap = 2LL * di->sm_count;
            const long long g = ra.n_items < cap ? ra.n_items : cap;
            R::compact_rope_kernel<<<(unsigned)g, R::kThreads, smem, s>>>(mk, mv, ra);
        } else
            sga::compact_kernel<__nv_bfloat16, false><<<grid, sga::kCompactThreads, 0, s>>>(a);
    } else {
        if (rope_smem > 48 * 1024) return SGA_ERR_UNSUPPORTED;
        if (c.rope)
            sga::compact_kernel<float, true><<<grid, sga::kCompactThreads, rope_smem, s>>>(a);
        else
            sga::compact_kernel<float, false><<<grid, sga::kCompactThreads, 0, s>>>(a);
    }
    if ((st = launch_status()) != SGA_OK) return st;
    sga::compact_finalize_kernel<<<BH, 128 * sga::kFinalizeRuns, 0, s>>>(plan->d_partials, plan->n_chunks, k_sum,
                                                                        v_sum);
    return launch_status();
}

sga_status sga_forward(sga_plan_t plan, const void* Q, const void* K, const void* V,
                       const void* K_S, const void* V_S, const float* k_sum, const float* v_sum,
                       void* O, float* lse, float scale, void* stream) {
    sga_status st = check_plan(plan);
    if (st != SGA_OK) return st;
    if (!Q || !K || !V || !K_S || !V_S || !k_sum || !v_sum || !O) return SGA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(K_S) || !aligned16(V_S) ||
        !aligned16(k_sum) || !aligned16(v_sum) || !aligned16(O) || (lse && !aligned16(lse)))
        return SGA_ERR_ALIGNMENT;
    if (!(scale > 0.f) || !std::isfinite(scale)) return SGA_ERR_INVALID_ARG;
    const sga_config& c = plan->cfg;
    AttnProblem pb;
    pb.dtype = c.dtype;
    pb.kernel = c.kernel;
    pb.n_seg = c.B * c.H;
    pb.seg_rows = plan->T;
    pb.kv_rows = plan->S;
    pb.Q = Q;
    pb.Kt = K_S;
    pb.Vt = V_S;
    pb.O = O;
    pb.lse = lse;
    pb.scale = scale;
    pb.ex.on = (c.diag || c.mean) && plan->D > 0;
    pb.ex.diag = c.diag;
    pb.ex.mean = c.mean;
    pb.ex.mean_mode = c.mean_mode;
    pb.ex.dropped = plan->D;
    pb.ex.T = plan->T;
    pb.ex.slot = plan->d_slot;
    pb.ex.K = K;
    pb.ex.V = V;
    pb.ex.k_sum = k_sum;
    pb.ex.v_sum = v_sum;
    pb.ex.rope = rope_args(plan);
    pb.bias = nullptr;
    pb.rope = c.rope != 0;
    pb.drop_kv = -1;
    return run_attention(pb, reinterpret_cast<cudaStream_t>(stream));
}

static sga_status plain_attention(int n_seg, long long seg_rows, long long kv_rows, int dtype, int kernel,
                                  const void* Q, const void* K, const void* V, const float* bias, void* O,
                                  float* lse, float scale, void* stream) {
    if (!Q || !K || !V || !O) return SGA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || (lse && !aligned16(lse)))
        return SGA_ERR_ALIGNMENT;
    if (!(scale > 0.f) || !std::isfinite(scale)) return SGA_ERR_INVALID_ARG;
    AttnProblem pb;
    std::memset(&pb, 0, sizeof(pb));
    pb.dtype = dtype;
    pb.kernel = kernel;
    pb.n_seg = n_seg;
    pb.seg_rows = seg_rows;
    pb.kv_rows = kv_rows;
    pb.Q = Q;
    pb.Kt = K;
    pb.Vt = V;
    pb.O = O;
    pb.lse = lse;
    pb.scale = scale;
    pb.ex.on = 0;
    pb.bias = bias;
    pb.rope = false;
    pb.drop_kv = -1;
    return run_attention(pb, reinterpret_cast<cudaStream_t>(stream));
}

sga_status sga_dense_forward(int B, int H, int64_t T, int head_dim, int dtype, int kernel,
                             const void* Q, const void* K, const void* V, void* O, float* lse,
                             float scale, void* stream) {
    if (B <= 0 || H <= 0 || T <= 0) return SGA_ERR_INVALID_ARG;
    sga_status st = check_common(dtype, head_dim, kernel);
    if (st != SGA_OK) return st;
    if ((long long)B * H > 0x7FFFFFFFLL || T > 0x7FFFFFFFLL) return SGA_ERR_UNSUPPORTED;
    return plain_attention(B * H, T, T, dtype, kernel, Q, K, V, nullptr, O, lse, scale, stream);
}

sga_status sga_frame_forward(int B, int H, int N, int L, int head_dim, int dtype, int kernel,
                             const void* Q, const void* K, const void* V, void* O, float* lse,
                             float scale, void* stream) {
    if (B <= 0 || H <= 0 || N <= 0 || L <= 0) return SGA_ERR_INVALID_ARG;
    sga_status st = check_common(dtype, head_dim, kernel);
    if (st != SGA_OK) return st;
    if ((long long)B * H * N > 0x7FFFFFFFLL) return SGA_ERR_UNSUPPORTED;
    return plain_attention(B * H * N, L, L, dtype, kernel, Q, K, V, nullptr, O, lse, scale, stream);
}

sga_status sga_bias_forward(int B, int H, int64_t Tq, int64_t Tk, int head_dim, int dtype, int kernel,
                            const void* Q, const void* K, const void* V, const float* bias, void* O,
                            float* lse, float scale, void* stream) {
    if (B <= 0 || H <= 0 || Tq <= 0 || Tk <= 0 || !bias) return SGA_ERR_INVALID_ARG;
    sga_status st = check_common(dtype, head_dim, kernel);
    if (st != SGA_OK) return st;
    if ((long long)B * H > 0x7FFFFFFFLL || Tq > 0x7FFFFFFFLL || Tk > 0x7FFFFFFFLL) return SGA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(bias) & 3u) != 0) return SGA_ERR_ALIGNMENT;
    return plain_attention(B * H, Tq, Tk, dtype, kernel, Q, K, V, bias, O, lse, scale, stream);
}

sga_status sga_rope2d(sga_plan_t plan, void* X, void* stream) {
    sga_status st = check_plan(plan);
    if (st != SGA_OK) return st;
    if (!X) return SGA_ERR_INVALID_ARG;
    if (!aligned16(X)) return SGA_ERR_ALIGNMENT;
    if (!plan->cfg.rope) return SGA_ERR_INVALID_ARG;
    const long long rows = (long long)plan->cfg.B * plan->cfg.H * plan->T;
    const long long blocks = (rows + 255) / 256;
    if (blocks > 0x7FFFFFFFLL) return SGA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (plan->cfg.dtype == SGA_BF16)
        sga::rope2d_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
            reinterpret_cast<__nv_bfloat16*>(X), rows, plan->T, rope_args(plan));
    else
        sga::rope2d_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<float*>(X), rows, plan->T,
                                                                     rope_args(plan));
    return launch_status();
}

}  // extern "C"

namespace {

sga_status merge_geom(const sga_merge_config* c, sga::MergeGeom* g) {
    if (!c) return SGA_ERR_INVALID_ARG;
    if (c->B <= 0 || c->H <= 0 || c->N <= 0 || c->grid_h <= 0 || c->grid_w <= 0 || c->n_special < 0 ||
        c->n_t <= 0 || c->n_s <= 0 || c->r_permille < 0 || c->r_permille > 1000)
        return SGA_ERR_INVALID_ARG;
    if (c->head_dim != 64) return SGA_ERR_UNSUPPORTED;
    if (c->dtype != SGA_BF16 && c->dtype != SGA_F32) return SGA_ERR_UNSUPPORTED;
    const long long P = (long long)c->grid_h * c->grid_w, L = c->n_special + P;
    if (L * c->N > 0x7FFFFFFFLL || (long long)c->n_t * (c->n_s < P ? c->n_s : P) > sga::kMergeMaxBlock)
        return SGA_ERR_UNSUPPORTED;
    g->N = c->N;
    g->L = (int)L;
    g->P = (int)P;
    g->n_special = c->n_special;
    g->n_t = c->n_t;
    g->n_s = (int)(c->n_s < P ? c->n_s : P);
    g->r_permille = c->r_permille;
    g->n_chunks = (c->N + c->n_t - 1) / c->n_t;
    g->n_windows = (int)((P + g->n_s - 1) / g->n_s);
    g->T = L * c->N;
    const int nf_last = c->N - (g->n_chunks - 1) * c->n_t;
    g->M = (long long)(g->n_chunks - 1) * sga::merge_chunk_size(*g, c->n_t) + sga::merge_chunk_size(*g, nf_last);
    if ((long long)c->B * c->H > 65535 || g->n_chunks > 65535) return SGA_ERR_UNSUPPORTED;
    return SGA_OK;
}

bool g_merge_smem_set[kMaxDevices][3];

}  // namespace

extern "C" {

sga_status sga_merge_size(const sga_merge_config* cfg, int64_t* M) {
    sga::MergeGeom g;
    sga_status st = merge_geom(cfg, &g);
    if (st != SGA_OK) return st;
    if (!M) return SGA_ERR_INVALID_ARG;
    *M = g.M;
    return SGA_OK;
}

sga_status sga_merge(const sga_merge_config* cfg, const void* X, const void* Y, void* X_m, void* Y_m,
                     float* log_g, int32_t* map, void* stream) {
    sga::MergeGeom g;
    sga_status st = merge_geom(cfg, &g);
    if (st != SGA_OK) return st;
    if (!X || !X_m || !map || (Y != nullptr) != (Y_m != nullptr)) return SGA_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(X_m) || (Y && (!aligned16(Y) || !aligned16(Y_m))) ||
        (reinterpret_cast<uintptr_t>(map) & 3u) || (reinterpret_cast<uintptr_t>(log_g) & 3u))
        return SGA_ERR_ALIGNMENT;
    int dev;
    if (current_device(&dev) != SGA_OK) return SGA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SGA_ERR_INVALID_ARG;
    const int di = cfg->dtype == SGA_BF16 ? 0 : 1;
    const int elem = di == 0 ? 2 : 4;
    const int nb_max = g.n_t * g.n_s;                   // entries of the largest block
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return SGA_ERR_CUDA;
    // bf16 blocks of at most 128 sources and 128 destinations match on the tensor cores (their
    // rows then live in shared memory as bf16 tiles only); other blocks on the CUDA cores
    const bool tc = di == 0 && (g.n_t - 1) * g.n_s <= sga::kTcMaxSrc && g.n_s <= sga::kTcMaxDst;
    const int ki = tc ? 2 : di;
    const int extra = tc ? sga::merge_tc_extra_bytes(g.n_s) : 0;
    // the values are staged in shared memory beside the keys when both fit
    const bool y_smem = Y != nullptr && sga::merge_smem_bytes(nb_max, elem, true, !tc) + extra <= optin;
    const int smem = sga::merge_smem_bytes(nb_max, elem, y_smem, !tc) + extra;
    if (smem > optin) return SGA_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (!g_merge_smem_set[dev][ki]) {
            const cudaError_t e =
                ki == 2 ? cudaFuncSetAttribute(sga::merge_kernel<__nv_bfloat16, true>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, optin)
                : ki == 0 ? cudaFuncSetAttribute(sga::merge_kernel<__nv_bfloat16, false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, optin)
                          : cudaFuncSetAttribute(sga::merge_kernel<float, false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
            if (e != cudaSuccess) return SGA_ERR_CUDA;
            g_merge_smem_set[dev][ki] = true;
        }
    }
    sga::MergeArgs a;
    a.g = g;
    a.X = X;
    a.Y = Y;
    a.Xm = X_m;
    a.Ym = Y_m;
    a.log_g = log_g;
    a.map = map;
    a.nb_max = nb_max;
    a.y_smem = y_smem ? 1 : 0;
    dim3 grid((unsigned)g.n_windows + 1, (unsigned)g.n_chunks, (unsigned)(cfg->B * cfg->H));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (tc)
        sga::merge_kernel<__nv_bfloat16, true><<<grid, sga::kMergeThreads, smem, s>>>(a);
    else if (di == 0)
        sga::merge_kernel<__nv_bfloat16, false><<<grid, sga::kMergeThreads, smem, s>>>(a);
    else
        sga::merge_kernel<float, false><<<grid, sga::kMergeThreads, smem, s>>>(a);
    return launch_status();
}

sga_status sga_unmerge(const sga_merge_config* cfg, const int32_t* map, const void* Y_m, void* Y, void* stream) {
    sga::MergeGeom g;
    sga_status st = merge_geom(cfg, &g);
    if (st != SGA_OK) return st;
    if (!map || !Y_m || !Y) return SGA_ERR_INVALID_ARG;
    if (!aligned16(Y_m) || !aligned16(Y) || (reinterpret_cast<uintptr_t>(map) & 3u)) return SGA_ERR_ALIGNMENT;
    const long long rows = (long long)cfg->B * cfg->H * g.T;
    const int vec = cfg->dtype == SGA_BF16 ? 8 : 16;
    const long long blocks = (rows * vec + 255) / 256;
    if (blocks > 0x7FFFFFFFLL) return SGA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cfg->dtype == SGA_BF16)
        sga::unmerge_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(map, Y_m, Y, g.T, g.M, rows);
    else
        sga::unmerge_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(map, Y_m, Y, g.T, g.M, rows);
    return launch_status();
}

sga_status sga_selftest_timeout(void* stream) {
    // a small dense problem on buffers of its own; the producer never loads key tile 1, so the
    // MMA warp's bounded wait for it expires, the CTA aborts (every role leaves its loop, drains
    // what is in flight, frees TMEM) and the kernel records SGA_ERR_TIMEOUT
    const long long T = 4 * 128;
    const size_t bytes = (size_t)T * 64 * 2;
    void* buf = nullptr;
    if (cudaMalloc(&buf, 4 * bytes) != cudaSuccess) return SGA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    sga_status st = cudaMemsetAsync(buf, 0, 4 * bytes, s) == cudaSuccess ? SGA_OK : SGA_ERR_CUDA;
    if (st == SGA_OK) {
        AttnProblem pb;
        std::memset(&pb, 0, sizeof(pb));
        pb.dtype = SGA_BF16;
        pb.kernel = SGA_KERNEL_TC;
        pb.n_seg = 1;
        pb.seg_rows = T;
        pb.kv_rows = T;
        pb.Q = buf;
        pb.Kt = static_cast<char*>(buf) + bytes;
        pb.Vt = static_cast<char*>(buf) + 2 * bytes;
        pb.O = static_cast<char*>(buf) + 3 * bytes;
        pb.scale = 0.125f;
        pb.ex.on = 0;
        pb.drop_kv = 1;
        st = run_attention(pb, s);
    }
    if (st == SGA_OK) st = sga_device_status(stream);       // expected: SGA_ERR_TIMEOUT
    cudaFree(buf);
    return st;
}

}  // extern "C"

struct sga_stream_s {
    uint32_t magic;
    sga_plan_t plan;                        // SGA layers; null for the plain kinds
    sga_plain_spec spec;                    // dense / frame-local / size-aware layers
    int device;
    int depth;
    size_t in_bytes;                        // one of Q, K, V, O (SGA layers)
    size_t q_bytes, kv_bytes, bias_bytes;   // plain layers: Q and O, K and V, the bias
    std::vector<void*> q, k, v, o, ks, vs, bias;   // per buffer set
    std::vector<float*> ksum, vsum;
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    std::vector<cudaEvent_t> kv_in, q_in, done, out_read;
    std::vector<char> used;
    long long next = 0;
};

namespace {

constexpr uint32_t kStreamMagic = 0x53474153u;   // "SGAS"

void stream_free(sga_stream_s* s) {
    if (s->h2d) cudaStreamSynchronize(s->h2d);
    if (s->comp) cudaStreamSynchronize(s->comp);
    if (s->d2h) cudaStreamSynchronize(s->d2h);
    for (auto* vec : {&s->q, &s->k, &s->v, &s->o, &s->ks, &s->vs, &s->bias})
        for (void* p : *vec) if (p) cudaFree(p);
    for (auto* vec : {&s->ksum, &s->vsum})
        for (float* p : *vec) if (p) cudaFree(p);
    for (auto* vec : {&s->kv_in, &s->q_in, &s->done, &s->out_read})
        for (cudaEvent_t e : *vec) if (e) cudaEventDestroy(e);
    if (s->h2d) cudaStreamDestroy(s->h2d);
    if (s->comp) cudaStreamDestroy(s->comp);
    if (s->d2h) cudaStreamDestroy(s->d2h);
    s->magic = 0;
    delete s;
}

sga_status check_stream(sga_stream_t s) {
    if (!s || s->magic != kStreamMagic) return SGA_ERR_INVALID_ARG;
    if (s->plan) return check_plan(s->plan);
    int dev;
    if (current_device(&dev) != SGA_OK) return SGA_ERR_CUDA;
    return dev == s->device ? SGA_OK : SGA_ERR_PLAN_MISMATCH;
}

sga_status check_plain_spec(const sga_plain_spec* p) {
    if (!p) return SGA_ERR_INVALID_ARG;
    if (p->kind != SGA_PLAIN_DENSE && p->kind != SGA_PLAIN_FRAME && p->kind != SGA_PLAIN_BIAS)
        return SGA_ERR_INVALID_ARG;
    if (p->B <= 0 || p->H <= 0 || p->Tq <= 0) return SGA_ERR_INVALID_ARG;
    if (p->kind == SGA_PLAIN_BIAS && p->Tk <= 0) return SGA_ERR_INVALID_ARG;
    if (p->kind == SGA_PLAIN_FRAME && (p->N <= 0 || p->L <= 0 || (int64_t)p->N * p->L != p->Tq))
        return SGA_ERR_INVALID_ARG;
    sga_status st = check_common(p->dtype, p->head_dim, p->kernel);
    if (st != SGA_OK) return st;
    if ((long long)p->B * p->H > 0x7FFFFFFFLL || p->Tq > 0x7FFFFFFFLL || p->Tk > 0x7FFFFFFFLL) return SGA_ERR_UNSUPPORTED;
    return SGA_OK;
}

}  // namespace

extern "C" {

sga_status sga_stream_create(sga_plan_t plan, int depth, sga_stream_t* out) {
    if (!plan || !out || depth < 1 || depth > 8) return SGA_ERR_INVALID_ARG;
    *out = nullptr;
    sga_status st = check_plan(plan);
    if (st != SGA_OK) return st;
    sga_stream_s* s = new (std::nothrow) sga_stream_s();
    if (!s) return SGA_ERR_CUDA;
    s->magic = kStreamMagic;
    s->plan = plan;
    std::memset(&s->spec, 0, sizeof(s->spec));
    s->device = plan->device;
    s->depth = depth;
    const size_t elem = plan->cfg.dtype == SGA_BF16 ? 2 : 4;
    const size_t bh = (size_t)plan->cfg.B * plan->cfg.H;
    s->in_bytes = bh * (size_t)plan->T * 64 * elem;
    const size_t ks_bytes = bh * (size_t)(plan->S > 0 ? plan->S : 1) * 64 * elem;
    const size_t sum_bytes = bh * 64 * sizeof(float);
    bool ok = true;
    auto alloc = [&](size_t bytes) -> void* {
        void* p = nullptr;
        if (ok && cudaMalloc(&p, bytes) != cudaSuccess) { ok = false; p = nullptr; }
        return p;
    };
    auto event = [&]() -> cudaEvent_t {
        cudaEvent_t e = nullptr;
        if (ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) { ok = false; e = nullptr; }
        return e;
    };
    for (int i = 0; i < depth; ++i) {
        s->q.push_back(alloc(s->in_bytes));
        s->k.push_back(alloc(s->in_bytes));
        s->v.push_back(alloc(s->in_bytes));
        s->o.push_back(alloc(s->in_bytes));
        s->ks.push_back(alloc(ks_bytes));
        s->vs.push_back(alloc(ks_bytes));
        s->ksum.push_back(static_cast<float*>(alloc(sum_bytes)));
        s->vsum.push_back(static_cast<float*>(alloc(sum_bytes)));
        s->kv_in.push_back(event());
        s->q_in.push_back(event());
        s->done.push_back(event());
        s->out_read.push_back(event());
        s->used.push_back(0);
    }
    if (ok && (cudaStreamCreateWithFlags(&s->h2d, cudaStreamNonBlocking) != cudaSuccess ||
               cudaStreamCreateWithFlags(&s->comp, cudaStreamNonBlocking) != cudaSuccess ||
               cudaStreamCreateWithFlags(&s->d2h, cudaStreamNonBlocking) != cudaSuccess))
        ok = false;
    if (!ok) {
        stream_free(s);
        cudaGetLastError();
        return SGA_ERR_CUDA;
    }
    *out = s;
    return SGA_OK;
}

sga_status sga_stream_submit(sga_stream_t s, const void* Q_host, const void* K_host, const void* V_host,
                             void* O_host, float scale) {
    sga_status st = check_stream(s);
    if (st != SGA_OK) return st;
    if (!s->plan) return SGA_ERR_INVALID_ARG;                // a plain stream takes sga_stream_submit_plain
    if (!Q_host || !K_host || !V_host || !O_host) return SGA_ERR_INVALID_ARG;
    if (!(scale > 0.f)) scale = 0.125f;
    const int i = (int)(s->next % s->depth);
    const size_t n = s->in_bytes;
    auto cu = [](cudaError_t e) { return e == cudaSuccess; };
    // inputs: the layer that last read this buffer set has finished; K and V first
    if (s->used[i] && !cu(cudaStreamWaitEvent(s->h2d, s->done[i], 0))) return SGA_ERR_CUDA;
    if (!cu(cudaMemcpyAsync(s->k[i], K_host, n, cudaMemcpyHostToDevice, s->h2d)) ||
        !cu(cudaMemcpyAsync(s->v[i], V_host, n, cudaMemcpyHostToDevice, s->h2d)) ||
        !cu(cudaEventRecord(s->kv_in[i], s->h2d)) ||
        !cu(cudaMemcpyAsync(s->q[i], Q_host, n, cudaMemcpyHostToDevice, s->h2d)) ||
        !cu(cudaEventRecord(s->q_in[i], s->h2d)))
        return SGA_ERR_CUDA;
    // compute: compaction once K and V are in, attention once Q is; O is free once the previous
    // output of this set has been copied out
    if (!cu(cudaStreamWaitEvent(s->comp, s->kv_in[i], 0))) return SGA_ERR_CUDA;
    if (s->used[i] && !cu(cudaStreamWaitEvent(s->comp, s->out_read[i], 0))) return SGA_ERR_CUDA;
    if ((st = sga_compact(s->plan, s->k[i], s->v[i], s->ks[i], s->vs[i], s->ksum[i], s->vsum[i], s->comp)) != SGA_OK)
        return st;
    if (!cu(cudaStreamWaitEvent(s->comp, s->q_in[i], 0))) return SGA_ERR_CUDA;
    if ((st = sga_forward(s->plan, s->q[i], s->k[i], s->v[i], s->ks[i], s->vs[i], s->ksum[i], s->vsum[i], s->o[i],
                          nullptr, scale, s->comp)) != SGA_OK)
        return st;
    if (!cu(cudaEventRecord(s->done[i], s->comp))) return SGA_ERR_CUDA;
    // output
    if (!cu(cudaStreamWaitEvent(s->d2h, s->done[i], 0)) ||
        !cu(cudaMemcpyAsync(O_host, s->o[i], n, cudaMemcpyDeviceToHost, s->d2h)) ||
        !cu(cudaEventRecord(s->out_read[i], s->d2h)))
        return SGA_ERR_CUDA;
    s->used[i] = 1;
    ++s->next;
    return SGA_OK;
}

sga_status sga_stream_create_plain(const sga_plain_spec* spec, int depth, sga_stream_t* out) {
    if (!out || depth < 1 || depth > 8) return SGA_ERR_INVALID_ARG;
    *out = nullptr;
    sga_status st = check_plain_spec(spec);
    if (st != SGA_OK) return st;
    int dev;
    if (current_device(&dev) != SGA_OK) return SGA_ERR_CUDA;
    sga_stream_s* s = new (std::nothrow) sga_stream_s();
    if (!s) return SGA_ERR_CUDA;
    s->magic = kStreamMagic;
    s->plan = nullptr;
    s->spec = *spec;
    if (spec->kind != SGA_PLAIN_BIAS) s->spec.Tk = spec->Tq;
    s->device = dev;
    s->depth = depth;
    const size_t elem = spec->dtype == SGA_BF16 ? 2 : 4;
    const size_t bh = (size_t)spec->B * spec->H;
    s->q_bytes = bh * (size_t)spec->Tq * 64 * elem;
    s->kv_bytes = bh * (size_t)s->spec.Tk * 64 * elem;
    s->bias_bytes = spec->kind == SGA_PLAIN_BIAS ? bh * (size_t)spec->Tk * sizeof(float) : 0;
    bool ok = true;
    auto alloc = [&](size_t bytes) -> void* {
        void* p = nullptr;
        if (ok && bytes > 0 && cudaMalloc(&p, bytes) != cudaSuccess) { ok = false; p = nullptr; }
        return p;
    };
    auto event = [&]() -> cudaEvent_t {
        cudaEvent_t e = nullptr;
        if (ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) { ok = false; e = nullptr; }
        return e;
    };
    for (int i = 0; i < depth; ++i) {
        s->q.push_back(alloc(s->q_bytes));
        s->k.push_back(alloc(s->kv_bytes));
        s->v.push_back(alloc(s->kv_bytes));
        s->o.push_back(alloc(s->q_bytes));
        s->bias.push_back(alloc(s->bias_bytes));
        s->kv_in.push_back(event());
        s->q_in.push_back(event());
        s->done.push_back(event());
        s->out_read.push_back(event());
        s->used.push_back(0);
    }
    if (ok && (cudaStreamCreateWithFlags(&s->h2d, cudaStreamNonBlocking) != cudaSuccess ||
               cudaStreamCreateWithFlags(&s->comp, cudaStreamNonBlocking) != cudaSuccess ||
               cudaStreamCreateWithFlags(&s->d2h, cudaStreamNonBlocking) != cudaSuccess))
        ok = false;
    if (!ok) {
        stream_free(s);
        cudaGetLastError();
        return SGA_ERR_CUDA;
    }
    *out = s;
    return SGA_OK;
}

sga_status sga_stream_submit_plain(sga_stream_t s, const void* Q_host, const void* K_host, const void* V_host,
                                   const float* bias_host, void* O_host, float scale) {
    sga_status st = check_stream(s);
    if (st != SGA_OK) return st;
    if (s->plan) return SGA_ERR_INVALID_ARG;                 // an SGA stream takes sga_stream_submit
    const sga_plain_spec& p = s->spec;
    if (!Q_host || !K_host || !V_host || !O_host || ((p.kind == SGA_PLAIN_BIAS) != (bias_host != nullptr)))
        return SGA_ERR_INVALID_ARG;
    if (!(scale > 0.f)) scale = 0.125f;
    const int i = (int)(s->next % s->depth);
    auto cu = [](cudaError_t e) { return e == cudaSuccess; };
    // inputs: the layer that last read this buffer set has finished; K, V (and the bias) first
    if (s->used[i] && !cu(cudaStreamWaitEvent(s->h2d, s->done[i], 0))) return SGA_ERR_CUDA;
    if (!cu(cudaMemcpyAsync(s->k[i], K_host, s->kv_bytes, cudaMemcpyHostToDevice, s->h2d)) ||
        !cu(cudaMemcpyAsync(s->v[i], V_host, s->kv_bytes, cudaMemcpyHostToDevice, s->h2d)) ||
        (bias_host && !cu(cudaMemcpyAsync(s->bias[i], bias_host, s->bias_bytes, cudaMemcpyHostToDevice, s->h2d))) ||
        !cu(cudaMemcpyAsync(s->q[i], Q_host, s->q_bytes, cudaMemcpyHostToDevice, s->h2d)) ||
        !cu(cudaEventRecord(s->q_in[i], s->h2d)))
        return SGA_ERR_CUDA;
    // compute once every input is in and the previous output of this set has been copied out
    if (!cu(cudaStreamWaitEvent(s->comp, s->q_in[i], 0))) return SGA_ERR_CUDA;
    if (s->used[i] && !cu(cudaStreamWaitEvent(s->comp, s->out_read[i], 0))) return SGA_ERR_CUDA;
    if (p.kind == SGA_PLAIN_DENSE)
        st = sga_dense_forward(p.B, p.H, p.Tq, p.head_dim, p.dtype, p.kernel, s->q[i], s->k[i], s->v[i], s->o[i],
                               nullptr, scale, s->comp);
    else if (p.kind == SGA_PLAIN_FRAME)
        st = sga_frame_forward(p.B, p.H, p.N, p.L, p.head_dim, p.dtype, p.kernel, s->q[i], s->k[i], s->v[i],
                               s->o[i], nullptr, scale, s->comp);
    else
        st = sga_bias_forward(p.B, p.H, p.Tq, p.Tk, p.head_dim, p.dtype, p.kernel, s->q[i], s->k[i], s->v[i],
                              static_cast<const float*>(s->bias[i]), s->o[i], nullptr, scale, s->comp);
    if (st != SGA_OK) return st;
    if (!cu(cudaEventRecord(s->done[i], s->comp))) return SGA_ERR_CUDA;
    if (!cu(cudaStreamWaitEvent(s->d2h, s->done[i], 0)) ||
        !cu(cudaMemcpyAsync(O_host, s->o[i], s->q_bytes, cudaMemcpyDeviceToHost, s->d2h)) ||
        !cu(cudaEventRecord(s->out_read[i], s->d2h)))
        return SGA_ERR_CUDA;
    s->used[i] = 1;
    ++s->next;
    return SGA_OK;
}

sga_status sga_stream_synchronize(sga_stream_t s) {
    sga_status st = check_stream(s);
    if (st != SGA_OK) return st;
    if (cudaStreamSynchronize(s->h2d) != cudaSuccess || cudaStreamSynchronize(s->comp) != cudaSuccess ||
        cudaStreamSynchronize(s->d2h) != cudaSuccess)
        return SGA_ERR_CUDA;
    return SGA_OK;
}

sga_status sga_stream_handles(sga_stream_t s, void** h2d, void** compute, void** d2h) {
    if (!s || s->magic != kStreamMagic) return SGA_ERR_INVALID_ARG;
    if (h2d) *h2d = s->h2d;
    if (compute) *compute = s->comp;
    if (d2h) *d2h = s->d2h;
    return SGA_OK;
}

void sga_stream_destroy(sga_stream_t s) {
    if (!s || s->magic != kStreamMagic) return;
    stream_free(s);
}

sga_status sga_last_device_status(sga_plan_t plan, void* stream) {
    sga_status st = check_plan(plan);
    if (st != SGA_OK) return st;
    return sga_device_status(stream);
}

sga_status sga_device_status(void* stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return SGA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, sga::g_status, sizeof(int)) != cudaSuccess) return SGA_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(sga::g_status, &zero, sizeof(int)) != cudaSuccess) return SGA_ERR_CUDA;
    }
    return (sga_status)v;
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// sga_compact_noalloc: the compaction for callers that cannot allocate device memory.
//
// Its only scratch -- the per-block partial sums of the dropped rows -- lives in the fixed
// array below, which every GPU that loads this library holds until the process exits.  In host
// code the array's name is a host-side stand-in, not a device address, so the address is looked
// up once per device (with that device current) and passed to the kernel.
constexpr long long kNoallocScratchFloats = 2LL * 1024 * 1024;   // 8 MiB: B*H*ceil(T/2048) <= 16384
static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchFloats];

namespace {

float* g_noalloc_ptr[kMaxDevices];
unsigned long long g_noalloc_ctx[kMaxDevices];   // id of the context the address belongs to
bool g_noalloc_ready[kMaxDevices];
std::mutex g_noalloc_mu;

// Unique id of the calling thread's current CUDA context (ids are never reused within a
// process, unlike context handles), or 0 when it cannot be read.
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch array on `dev` (current).  It is looked up with the device
// current and cached per device together with the id of the context it was looked up in: after
// a device reset (or any new primary context) the library's module is loaded again at another
// address, so a changed context id triggers a fresh lookup.  No allocation is made.
sga_status noalloc_scratch(int dev, float** out) {
    if (dev < 0 || dev >= kMaxDevices) return SGA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    const unsigned long long ctx = current_context_id();
    if (!g_noalloc_ready[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
        float* p = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_noalloc_scratch) != cudaSuccess || !p)
            return SGA_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
        // the lookup made the primary context current if it was not: read its id now
        g_noalloc_ctx[dev] = ctx != 0 ? ctx : current_context_id();
        g_noalloc_ready[dev] = true;
    }
    *out = g_noalloc_ptr[dev];
    return SGA_OK;
}

// |S| of a configuration in closed form (no allocation): per frame, L tokens when the frame is
// kept whole, else the special tokens plus ceil((G_h - phi_r)/s_h) * ceil((G_w - phi_c)/s_w).
long long kept_count_closed_form(const sga_config& c) {
    const long long L = (long long)c.n_special + (long long)c.grid_h * c.grid_w;
    long long total = 0;
    for (int f = 0; f < c.N; ++f) {
        if ((f == 0 && c.ref_frame_dense) || (c.s_h == 1 && c.s_w == 1)) {
            total += L;
            continue;
        }
        const int pr = c.phase_shift ? (f / c.s_w) % c.s_h : 0;
        const int pc = c.phase_shift ? f % c.s_w : 0;
        const long long rows = pr < c.grid_h ? (c.grid_h - pr + c.s_h - 1) / c.s_h : 0;
        const long long cols = pc < c.grid_w ? (c.grid_w - pc + c.s_w - 1) / c.s_w : 0;
        total += c.n_special + rows * cols;
    }
    return total;
}

}  // namespace

extern "C" sga_status sga_kept_count(const sga_config* cfg, int64_t* S) {
    if (!S) return SGA_ERR_INVALID_ARG;
    sga_status st = check_config(cfg);
    if (st != SGA_OK) return st;
    *S = kept_count_closed_form(*cfg);
    return SGA_OK;
}

extern "C" sga_status sga_compact_noalloc(const sga_config* cfg, const void* K, const void* V, void* K_S,
                                          void* V_S, float* k_sum, float* v_sum, void* stream) {
    sga_status st = check_config(cfg);
    if (st != SGA_OK) return st;
    if (cfg->rope) return SGA_ERR_UNSUPPORTED;
    if (!K || !V || !K_S || !V_S || !k_sum || !v_sum) return SGA_ERR_INVALID_ARG;
    if (!aligned16(K) || !aligned16(V) || !aligned16(K_S) || !aligned16(V_S) || !aligned16(k_sum) ||
        !aligned16(v_sum))
        return SGA_ERR_ALIGNMENT;
    const sga_config& c = *cfg;
    const long long L = (long long)c.n_special + (long long)c.grid_h * c.grid_w;
    const long long T = L * c.N;
    const long long BH = (long long)c.B * c.H;
    const long long n_chunks = (T + kCompactRowsPerChunk - 1) / kCompactRowsPerChunk;
    if (BH > 65535 || n_chunks > 0x7FFFFFFFLL) return SGA_ERR_UNSUPPORTED;
    if (BH * n_chunks * 128 > kNoallocScratchFloats) return SGA_ERR_SCRATCH_LIMIT;
    int dev;
    if (current_device(&dev) != SGA_OK) return SGA_ERR_CUDA;
    float* scratch = nullptr;
    if ((st = noalloc_scratch(dev, &scratch)) != SGA_OK) return st;

    sga::NoallocArgs a;
    a.T = T;
    a.S = kept_count_closed_form(c);
    a.L = (int)L;
    a.n_special = c.n_special;
    a.grid_h = c.grid_h;
    a.grid_w = c.grid_w;
    a.s_h = c.s_h;
    a.s_w = c.s_w;
    a.phase_shift = c.phase_shift;
    a.ref_frame_dense = c.ref_frame_dense;
    a.rows_per_chunk = kCompactRowsPerChunk;
    a.n_chunks = (int)n_chunks;
    a.K = K;
    a.V = V;
    a.KS = K_S;
    a.VS = V_S;
    a.partials = scratch;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    dim3 grid((unsigned)n_chunks, (unsigned)BH);
    if (c.dtype == SGA_BF16)
        sga::compact_noalloc_kernel<__nv_bfloat16><<<grid, sga::kCompactThreads, 0, s>>>(a);
    else
        sga::compact_noalloc_kernel<float><<<grid, sga::kCompactThreads, 0, s>>>(a);
    if ((st = launch_status()) != SGA_OK) return st;
    sga::compact_finalize_kernel<<<(unsigned)BH, 128 * sga::kFinalizeRuns, 0, s>>>(scratch, (int)n_chunks, k_sum,
                                                                                  v_sum);
    return launch_status();
}
