/*
 * sga.h -- C ABI of libsga: Subsampling Global Attention (SGA) for one global cross-frame
 * attention layer of a VGGT-style multi-view transformer, on one B300 GPU (sm_103a).
 *
 * The method (sources are web pages, cited by title and section):
 *   "AVGGT: Rethinking Global Attention for Accelerating VGGT" (CVPR 2026 notes)
 *     Key design 1  Global-to-Frame: a global layer may run as attention within each frame.
 *     Key design 2  SGA: every query is kept; keys/values are cut to a grid subset S -- the
 *                   first patch token of each s_h x s_w window (sigma = s_h*s_w; 2->(1,2),
 *                   4->(2,2), 6->(2,3), 9->(3,3)); special tokens and, for VGGT, frame 0
 *                   stay uncompressed.  Standard attention softmax(QK^T/sqrt(d))V over S.
 *     Key design 3  two more components disjoint from S under the same softmax: each token's
 *                   own key (diagonal) and one mean key/value for all dropped patches.
 *   "RegimeVGGT: Layer-Wise Spatially Preserving Redundancy Removal for Visual Geometry
 *    Grounded Transformer" (NeurIPS 2026 notes)
 *     Core mechanism  L = T + 5 tokens per frame (patches + 5 camera/register tokens).
 *     Key design 2    size-aware attention softmax(QK^T/sqrt(d) + log g^T)V: a key that
 *                     stands for g tokens gets the logit bias ln g (here: the mean key,
 *                     g = number of dropped tokens it averages).
 *     Key design 3    per-frame phase shift of the grid (row (f div t) mod t, column
 *                     f mod t); frame 0 and camera/register tokens at full density.
 *
 * Readings where the pages are silent (identical in the library and its test oracle):
 *   special tokens are the first n_special slots of each frame, patches follow row-major;
 *   partial edge windows keep their top-left token; for a (s_h, s_w) grid the phase is
 *   row (f div s_w) mod s_h, column f mod s_w; the diagonal term exists only for a dropped
 *   query; the mean is leave-one-out for a dropped query (mean over D \ {i}, count c-1)
 *   unless SGA_MEAN_GLOBAL is chosen; the bias is + ln(count) after the 1/sqrt(d) scaling;
 *   the mean runs over every dropped token of all frames of one (batch, head).
 *
 * Tensors.  Q, K, V, O are contiguous [B, H, T, 64] with T = N*L tokens (token t = f*L + p),
 * in the dtype of the call (SGA_BF16: bfloat16; SGA_F32: float32).  All pointers are DEVICE
 * pointers owned by the caller and must stay valid until the stream reaches the work; each
 * must be 16-byte aligned.  Calls never allocate, never synchronise the host (except
 * sga_device_status) and enqueue their kernels on `stream` (a cudaStream_t; NULL = the legacy
 * default stream) of the device that is current on the calling thread.
 *
 * Errors.  Every call validates its arguments first and returns a status; nothing aborts or
 * traps.  Kernels that wait on hardware barriers give up after a bounded time, record
 * SGA_ERR_TIMEOUT in a device status word and return; sga_device_status() reads it.
 */
#ifndef SGA_H_
#define SGA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SGA_OK = 0,
    SGA_ERR_INVALID_ARG = 1,    /* null pointer, non-positive size, inconsistent shape */
    SGA_ERR_UNSUPPORTED = 2,    /* head_dim != 64, unknown dtype, kernel not built for it */
    SGA_ERR_ALIGNMENT = 3,      /* a tensor pointer is not 16-byte aligned */
    SGA_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed (launch, memcpy, ...) */
    SGA_ERR_TIMEOUT = 5,        /* a kernel's bounded wait expired (reported by device status) */
    SGA_ERR_PLAN_MISMATCH = 6,  /* plan used with another device or a destroyed plan */
    SGA_ERR_SCRATCH_LIMIT = 7,  /* problem larger than sga_compact_noalloc's fixed scratch */
    SGA_ERR_DEBUG_CHECK = 8     /* debug builds only: a kernel's index check failed (access skipped) */
} sga_status;

typedef enum { SGA_BF16 = 0, SGA_F32 = 1 } sga_dtype;

/* Mean-term reading (see above).  LOO keeps S, {i} and D\{i} disjoint for every query. */
typedef enum { SGA_MEAN_LOO = 0, SGA_MEAN_GLOBAL = 1 } sga_mean_mode;

/* Which attention kernel runs.  AUTO: tensor-core kernel (tcgen05/TMEM/TMA) for bf16,
 * CUDA-core fp32 kernel for f32.  SIMT forces the CUDA-core kernel (any dtype). */
typedef enum { SGA_KERNEL_AUTO = 0, SGA_KERNEL_TC = 1, SGA_KERNEL_SIMT = 2 } sga_kernel;

/* Layer configuration.  L = n_special + grid_h*grid_w tokens per frame, T = N*L. */
typedef struct {
    int B, H;                /* batch elements, heads */
    int N;                   /* frames */
    int grid_h, grid_w;      /* patch grid of one frame */
    int n_special;           /* camera/register tokens per frame (VGGT: 5) */
    int head_dim;            /* must be 64 */
    int s_h, s_w;            /* subsampling window, sigma = s_h*s_w; (1,1) keeps every key */
    int phase_shift;         /* 1: per-frame phase-shifted grid */
    int ref_frame_dense;     /* 1: frame 0 uncompressed (VGGT); 0: all frames alike (pi^3) */
    int diag;                /* 1: diagonal self term for dropped queries */
    int mean;                /* 1: log(count)-biased mean key/value of the dropped set */
    int mean_mode;           /* sga_mean_mode */
    int dtype;               /* sga_dtype of Q, K, V, O, K_S, V_S */
    int kernel;              /* sga_kernel */
    /* 2D rotary position embedding of Q and K, fused into the layer (VGGT re-applies RoPE in
     * every layer: "HTTM: Head-wise Temporal Token Merging for Faster VGGT", section 3).  The
     * pages give no convention; the one used: head dims [0, 32) rotate by the row position,
     * [32, 64) by the column position; in each half the pairs (j, j+16), j < 16, rotate by
     * pos * rope_base^(-j/16); a patch (r, c) sits at (r + rope_pos_offset, c + rope_pos_offset),
     * the n_special tokens at position 0 (not rotated).  With rope = 1, sga_compact writes the
     * rotated kept keys and sums the rotated dropped keys, and sga_forward rotates Q and the
     * diagonal / leave-one-out keys itself: K and Q in memory stay unrotated.  V is never
     * rotated. */
    int rope;                /* 0: off, 1: on */
    float rope_base;         /* frequency base (> 1) */
    int rope_pos_offset;     /* >= 0 */
} sga_config;

typedef struct sga_plan_s* sga_plan_t;   /* opaque */

/* Host-only plan builder: the same kept set S as sga_plan_create, computed on the host without
 * touching any device.  kv_index (capacity T = N*L entries) receives the kept tokens in
 * ascending order, frame_off (N+1 entries) each frame's first index into kv_index, slot
 * (T entries, nullable) the position of each token in kv_index or -1 if dropped, *S_out |S|.
 * Source: AVGGT Key design 2; RegimeVGGT Key design 3. */
sga_status sga_plan_host(const sga_config* cfg, int32_t* kv_index, int32_t* frame_off,
                         int32_t* slot, int64_t* S_out);

/* Generalised kept-set description ("RegimeVGGT ..." Key design 3): per-axis window sizes that
 * need not be integers, given exactly as rationals sigma = num/den >= 1 (1.5 = 3/2, 1.3 = 13/10,
 * 1.7 = 17/10).  Along an axis of length G, window i covers [i*sigma, (i+1)*sigma) and keeps
 * its first position ceil(i*sigma), about G/sigma positions.  With phase_shift the positions
 * move by phi_r = (f div t_w) mod t_h, phi_c = f mod t_w, t = ceil(sigma) per axis (the page's
 * formula with an integer tile).  Integer sigma gives exactly the AVGGT grid of
 * sga_plan_host / sga_plan_create. */
typedef struct {
    int N, grid_h, grid_w, n_special;
    int sh_num, sh_den;      /* row window sigma_h = sh_num / sh_den */
    int sw_num, sw_den;      /* column window sigma_w = sw_num / sw_den */
    int phase_shift, ref_frame_dense;
} sga_grid_spec;

/* Host-only builder of the generalised kept set: frame 0 (when dense), the camera/register
 * tokens, the window starts above, and every token of protected_tokens (host int32
 * [n_protected], any order, repeats allowed -- e.g. the salient tokens RegimeVGGT protects).
 * Outputs as sga_plan_host (kv_index capacity N*L).  SGA_ERR_INVALID_ARG for a protected index
 * outside [0, N*L). */
sga_status sga_plan_host_general(const sga_grid_spec* spec, const int32_t* protected_tokens, int64_t n_protected,
                                 int32_t* kv_index, int32_t* frame_off, int32_t* slot, int64_t* S_out);

/* A plan from an arbitrary kept set: `kv_index` (host int32 [S], strictly ascending tokens in
 * [0, T), T = N*L from cfg) replaces the grid rule; cfg's s_h, s_w and phase_shift are not used,
 * everything else (B, H, frame geometry, diag, mean, dtype, kernel) is.  The same compaction and
 * attention run on it; the dropped set D is the complement of kv_index.  Allocates like
 * sga_plan_create.  SGA_ERR_INVALID_ARG if the list is not strictly ascending or out of range. */
sga_status sga_plan_create_from_index(const sga_config* cfg, const int32_t* kv_index, int64_t S, int device,
                                      sga_plan_t* out);

/* Build the kept set S for `cfg` on the host (integer arithmetic, O(T)) and upload it to
 * `device`: the token->slot map (int32 [T], -1 = dropped), the kept-token list (int32 [|S|],
 * ascending) and per-frame offsets (int32 [N+1]).  The plan owns these device buffers and a
 * small reduction scratch buffer; sga_plan_destroy frees them.  This is the only call that
 * allocates (cudaMalloc) and it synchronises `device` once after the upload.
 * Source: AVGGT Key design 2; RegimeVGGT Key design 3. */
sga_status sga_plan_create(const sga_config* cfg, int device, sga_plan_t* out);

/* T = N*L, S = |S| (kept keys), dropped = T - |S|.  Any output pointer may be NULL. */
sga_status sga_plan_info(sga_plan_t plan, int64_t* T, int64_t* S, int64_t* dropped);

/* Copy the plan's kept-token list (host int32 [|S|]) and frame offsets (host int32 [N+1]).
 * Either pointer may be NULL.  Synchronous. */
sga_status sga_plan_copy_indices(sga_plan_t plan, int32_t* kv_index, int32_t* frame_off);

/* Free the plan's device buffers (synchronises the plan's device).  NULL is a no-op. */
void sga_plan_destroy(sga_plan_t plan);

/* Compaction (AVGGT Key design 2 "replace K, V by the subset S" and Key design 3 "one mean
 * key/value for all dropped patches"): K_S, V_S [B, H, |S|, 64] receive exact copies of the
 * kept rows of K, V [B, H, T, 64] in ascending token order; k_sum, v_sum (fp32 [B, H, 64])
 * receive the sums of the dropped rows (a fixed-order, deterministic reduction).  The mean
 * is formed from these sums by sga_forward.  Uses the plan's scratch buffer: two calls with
 * the same plan must not run concurrently on different streams. */
sga_status sga_compact(sga_plan_t plan, const void* K, const void* V, void* K_S, void* V_S,
                       float* k_sum, float* v_sum, void* stream);

/* SGA attention (AVGGT Key designs 2-3, RegimeVGGT Key design 2).  For every query row i of
 * every (b, h):  O_i = softmax over { scale*q_i.k_j : j in S }
 *                                 U { scale*q_i.k_i           if diag and i dropped }
 *                                 U { scale*q_i.kbar_i + ln c_i  if mean and c_i > 0 }
 * applied to the matching values, where kbar_i, vbar_i, c_i are the mean key/value and count
 * of the dropped set (leave-one-out for a dropped i under SGA_MEAN_LOO), formed from k_sum,
 * v_sum.  Q, K, V: [B, H, T, 64]; K_S, V_S, k_sum, v_sum from sga_compact with this plan.
 * O: [B, H, T, 64] (RN-even from fp32).  lse: optional fp32 [B, H, T], natural-log
 * log-sum-exp of each row's logits (NULL to skip).  scale: the logit scale (1/sqrt(64)). */
sga_status sga_forward(sga_plan_t plan, const void* Q, const void* K, const void* V,
                       const void* K_S, const void* V_S, const float* k_sum, const float* v_sum,
                       void* O, float* lse, float scale, void* stream);

/* Dense global attention, softmax(scale*QK^T)V over all T tokens of each (b, h)
 * (AVGGT Key design 2, the standard attention equation; SGA with sigma = 1). */
sga_status sga_dense_forward(int B, int H, int64_t T, int head_dim, int dtype, int kernel,
                             const void* Q, const void* K, const void* V, void* O, float* lse,
                             float scale, void* stream);

/* Frame-local attention (AVGGT Key design 1, Global-to-Frame): each query attends to the L
 * tokens of its own frame only; Q, K, V, O are [B, H, N*L, 64]. */
sga_status sga_frame_forward(int B, int H, int N, int L, int head_dim, int dtype, int kernel,
                             const void* Q, const void* K, const void* V, void* O, float* lse,
                             float scale, void* stream);

/* Size-aware attention ("RegimeVGGT ..." Key design 2): for every query row of every (b, h),
 *   O_i = softmax over j of ( scale * q_i . k_j + bias_j ) applied to v_j,
 * where bias_j is the natural-log bias of key j -- ln g_j for a key that stands for g_j source
 * tokens (g_j = 1: bias 0), or any real value.  Q: [B, H, Tq, 64]; K, V: [B, H, Tk, 64];
 * bias: fp32 [B, H, Tk] (4-byte aligned device pointer); O: [B, H, Tq, 64]; lse: optional fp32
 * [B, H, Tq].  The tensor-core kernel adds the bias inside the QK^T product (an extra K step
 * holding bias/scale in two bf16 parts, about 2^-16 relative precision); the CUDA-core kernel
 * adds it in fp32.  Same conventions and errors as sga_dense_forward. */
sga_status sga_bias_forward(int B, int H, int64_t Tq, int64_t Tk, int head_dim, int dtype, int kernel,
                            const void* Q, const void* K, const void* V, const float* bias, void* O,
                            float* lse, float scale, void* stream);

/* Rotate X [B, H, T, 64] (the plan's shape and dtype) in place with the plan's 2D rotary
 * embedding (cfg.rope must be 1): for a dense or frame-local layer with RoPE, rotate Q and K with
 * this call, then call sga_dense_forward / sga_frame_forward.  HBM-bound, one pass. */
sga_status sga_rope2d(sga_plan_t plan, void* X, void* stream);

/* Head-wise temporal token merging ("HTTM: Head-wise Temporal Token Merging for Faster VGGT",
 * section 2; "RegimeVGGT ..." Key designs 1-2).  Every (batch, head) merges its own tokens:
 *   - frames are grouped in chunks of n_t; a block is the run of n_s consecutive patch tokens
 *     (row-major; the last run of a frame may be shorter) in every frame of one chunk;
 *     n_t * min(n_s, grid_h*grid_w) <= 512;
 *   - the chunk's first frame holds the destinations (first-frame anchoring), the other frames
 *     the sources; special tokens are never merged;
 *   - each source joins the destination of its block with the largest cosine similarity of X
 *     (first maximum), and the floor(#sources * r_permille / 1000) most similar sources of the
 *     block are merged (ties: lower token index); the cosine is decided in IEEE fp32 with one
 *     fixed order (fma chains over the 64 dims, correctly rounded sqrt and division);
 *   - a merged token is the mean of its members; Y (values) follows X's matching.
 * The merged sequence (M tokens per (b, h), sga_merge_size) is block-major: for each chunk its
 * special tokens, then each window's kept tokens (destinations and unmerged sources), in token
 * order.  map[t] is the merged index that token t belongs to, log_g (nullable) the natural log
 * of each merged token's group size -- the bias of sga_bias_forward (size-aware attention).
 * X [B, H, N*L, 64]; Y nullable (then Y_m must be null); X_m, Y_m [B, H, M, 64];
 * log_g fp32 [B, H, M]; map int32 [B, H, N*L]. */
typedef struct {
    int B, H, N, grid_h, grid_w, n_special, head_dim;
    int n_t;                 /* frames per chunk (temporal block depth) */
    int n_s;                 /* patch tokens per spatial run */
    int r_permille;          /* share of a block's sources merged, in 1/1000 */
    int dtype;               /* sga_dtype */
} sga_merge_config;

sga_status sga_merge_size(const sga_merge_config* cfg, int64_t* M);
sga_status sga_merge(const sga_merge_config* cfg, const void* X, const void* Y, void* X_m, void* Y_m,
                     float* log_g, int32_t* map, void* stream);

/* Unmerge: Y[b, h, t] = Y_m[b, h, map[b, h, t]] -- every token receives the output of the
 * merged token it belongs to (merged queries' attention outputs copied back). */
sga_status sga_unmerge(const sga_merge_config* cfg, const int32_t* map, const void* Y_m, void* Y, void* stream);

/* Compaction that allocates nothing, for callers that cannot call cudaMalloc.  The pages have
 * no counterpart: this entry point exists for integration only.
 *
 * Who needs it: code that runs where device allocation is off limits -- for example, inside
 * an engine whose memory is fully reserved up front by its own allocator, a plug-in that the
 * host framework forbids to allocate, or a step that must not pay for (or risk failing) an
 * allocation.  Such a caller cannot create an sga_plan_t (sga_plan_create allocates the plan's
 * index buffers and scratch).  This call needs no plan: it derives each token's place in K_S
 * from `cfg` in closed form and keeps its only scratch -- the per-block partial sums of the
 * dropped rows -- in a fixed array inside the library.
 *
 * Results are those of sga_compact with a plan for `cfg`: K_S, V_S [B, H, |S|, 64] get the
 * kept rows of K, V [B, H, T, 64] in ascending token order, and k_sum, v_sum (fp32 [B, H, 64])
 * get the sums of the dropped rows.  |S| comes from sga_kept_count (or sga_plan_host /
 * sga_plan_info); the call receives no buffer sizes, so the caller must size K_S and V_S by
 * it (the Python binding checks this before the call).  All pointers are caller-owned device
 * memory, 16-byte aligned.  No cudaMalloc, cudaFree or other allocating call is made.
 *
 * No rotary embedding: a configuration with rope = 1 returns SGA_ERR_UNSUPPORTED.
 *
 * Limit: B * H * ceil(T / 2048) <= 16384 (the scratch holds 2^21 floats, 8 MiB, which every
 * GPU that loads the library keeps until the process exits); larger problems return
 * SGA_ERR_SCRATCH_LIMIT before anything is launched.  A layer of 800 frames of 1374 tokens
 * with 16 heads (T = 1,099,200) needs 8592.
 *
 * The first call on a device looks up the scratch array's device address (once per device,
 * with that device current); make that first call before any stream capture.  The address is
 * cached with the id of the context it belongs to: after a device reset (a new primary context)
 * the next call looks it up again.  Every call on a device shares the one scratch array, so
 * calls that may overlap on the GPU (other streams, other host threads) race and must be
 * serialised by the caller.  The array keeps the last
 * call's contents; nothing in it needs to start at zero because each call overwrites every
 * partial it reads. */
sga_status sga_compact_noalloc(const sga_config* cfg, const void* K, const void* V, void* K_S,
                               void* V_S, float* k_sum, float* v_sum, void* stream);

/* |S| of `cfg` in closed form (host only, allocates nothing): per frame, L tokens when the frame
 * is kept whole, else n_special + ceil((grid_h - phi_r) / s_h) * ceil((grid_w - phi_c) / s_w)
 * with the frame's phase (phi_r, phi_c).  Equals sga_plan_info's S for a plan of `cfg`.  The
 * buffers K_S and V_S given to sga_compact_noalloc must hold exactly this many rows per (b, h):
 * the call receives no sizes and cannot check them itself.  SGA_ERR_INVALID_ARG for a bad
 * configuration or a NULL S. */
sga_status sga_kept_count(const sga_config* cfg, int64_t* S);

/* Streaming from host memory (no counterpart on the pages; the executor that feeds the layer
 * from host buffers).  A stream object owns, for one plan, `depth` sets of device tensors (Q, K,
 * V, O, K_S, V_S and the two sums) and three CUDA streams of its own: host-to-device copies,
 * compute, device-to-host copies.  Every device allocation happens in sga_stream_create.
 *
 * sga_stream_submit queues one whole layer: copies K and V, then Q, from the HOST pointers
 * into the next buffer set, runs sga_compact as soon as K and V have arrived and sga_forward
 * once Q has, and copies O back to the host pointer.  It returns at once.  Consecutive submits
 * overlap: layer i+1's inputs and layer i-1's output move while layer i computes.  Events order
 * every reuse of a buffer set after the work that last read it, so each output equals
 * sga_compact + sga_forward on the same inputs.  Host buffers are [B, H, T, 64] in the plan's
 * dtype; they must stay valid and unchanged until sga_stream_synchronize returns, and they
 * should be page-locked (cudaHostAlloc / cudaHostRegister) for the copies to overlap.
 * `scale` <= 0 means 1/sqrt(64).  All calls need the plan's device current; the plan must
 * outlive the stream object.  depth: 1 .. 8 buffer sets. */
typedef struct sga_stream_s* sga_stream_t;
sga_status sga_stream_create(sga_plan_t plan, int depth, sga_stream_t* out);
sga_status sga_stream_submit(sga_stream_t s, const void* Q_host, const void* K_host, const void* V_host,
                             void* O_host, float scale);
/* The same executor for the plain attention calls: dense global attention (sga_dense_forward),
 * frame-local attention (sga_frame_forward) and size-aware attention (sga_bias_forward).
 * spec->kind picks the call; B, H, head_dim, dtype and kernel are its arguments; Tq is the query
 * (and output) rows per (b, h); Tk the key rows (SGA_PLAIN_BIAS only, else Tq is used); N and L
 * the frames and tokens per frame (SGA_PLAIN_FRAME only, N*L = Tq).  A stream object made here
 * takes sga_stream_submit_plain (sga_stream_submit refuses it, and the other way round); it
 * uses the device current at creation.  sga_stream_submit_plain copies K, V, the bias (host fp32
 * [B, H, Tk]; SGA_PLAIN_BIAS only, else NULL) and Q in, runs the call once they have arrived and
 * copies O [B, H, Tq, 64] back, overlapping consecutive submits like sga_stream_submit. */
typedef enum { SGA_PLAIN_DENSE = 1, SGA_PLAIN_FRAME = 2, SGA_PLAIN_BIAS = 3 } sga_plain_kind;
typedef struct {
    int kind;                /* sga_plain_kind */
    int B, H;
    int64_t Tq, Tk;
    int N, L;
    int head_dim, dtype, kernel;
} sga_plain_spec;
sga_status sga_stream_create_plain(const sga_plain_spec* spec, int depth, sga_stream_t* out);
sga_status sga_stream_submit_plain(sga_stream_t s, const void* Q_host, const void* K_host, const void* V_host,
                                   const float* bias_host, void* O_host, float scale);
/* Wait until every submitted layer's output is in its host buffer. */
sga_status sga_stream_synchronize(sga_stream_t s);
/* The object's CUDA streams (cudaStream_t), e.g. to record timing events around submits:
 * h2d receives the first work of a submit, d2h the last. */
sga_status sga_stream_handles(sga_stream_t s, void** h2d, void** compute, void** d2h);
/* Waits for outstanding work, then frees everything the object owns.  NULL is a no-op. */
void sga_stream_destroy(sga_stream_t s);

/* Synchronise `stream`, then read and clear the device status word of the current device
 * (SGA_OK or SGA_ERR_TIMEOUT from a kernel's bounded wait).  Returns SGA_ERR_CUDA if the
 * synchronisation itself failed. */
sga_status sga_device_status(void* stream);

/* The same read for the device of `plan` (which must be current): SGA_ERR_PLAN_MISMATCH for an
 * invalid plan or another current device, else the result of sga_device_status(stream).  The
 * status word is per device, not per plan: it reports every library kernel that ran on the
 * device since the last read. */
sga_status sga_last_device_status(sga_plan_t plan, void* stream);

/* Failure-detection self-test of the bounded waits (no counterpart on the pages; it checks
 * the error path of this library).  Runs the tensor-core attention kernel on a small dense
 * problem (buffers of its own, allocated and freed here) in which the TMA producer never loads
 * one key tile, so nothing ever completes that tile's barrier.  The MMA warp's bounded wait
 * expires (about 2 s of SM clocks), the CTA aborts -- every role leaves its loop, waits (again
 * bounded) for the copies and products already in flight, frees its Tensor Memory and returns
 * -- and the kernel records SGA_ERR_TIMEOUT.  Synchronises `stream` and returns the status it
 * read (and cleared): SGA_ERR_TIMEOUT when the mechanism works.  The context stays usable. */
sga_status sga_selftest_timeout(void* stream);

/* Debug builds of the library (compiled with -DSGA_DEBUG; sga_build_info then contains "debug")
 * check every indexed store of the compaction, attention, merge and unmerge kernels, and the
 * index reads that steer them, against the buffer's bound; a failed check skips the access,
 * sets the device status word to SGA_ERR_DEBUG_CHECK and records the first failure.  This call
 * copies that record to the host and clears it: `site` (the check that failed: 1-3 compaction,
 * 10-12 attention, 20-23 merging), the offending `index`, its `bound`, and `count`, the number of
 * failed checks.  Any output pointer may be NULL.  Synchronous.  A normal build returns
 * SGA_ERR_UNSUPPORTED. */
sga_status sga_debug_report(int64_t* site, int64_t* index, int64_t* bound, int64_t* count);

/* Static description of a status code. */
const char* sga_status_string(sga_status s);

/* Library build identification: compute capability targeted ("sm_103a"), version, and
 * "src=<fingerprint>" of the sources it was compiled from (the build passes SGA_SOURCE_HASH). */
const char* sga_build_info(void);

#ifdef __cplusplus
}
#endif
#endif /* SGA_H_ */
