/*
 * ssd.h -- C ABI of libssd: the Mamba-2 SSD chunked selective scan on one
 * GB300 (sm_103a).
 *
 * The operation (forward): for every batch b and head h, with g(h) = h/(H/G)
 *     delta_t = softplus(dt[b,t,h] + dt_bias[h])          (softplus(v) = v for v > 20)
 *     h_t     = exp(delta_t * A[h]) * h_{t-1} + delta_t * x_t (outer) B_t[g(h)]
 *     y_t     = C_t[g(h)] . h_t + D[h] * x_t,     h_{-1} = init,  final = h_{T-1}
 * computed by the chunked algorithm of the pages: chunk_cumsum, chunk_state,
 * state_passing and chunk_scan ("Optimizing Mamba-2 kernels for the B200",
 * Stage 1 kernel table, fwd_2 / fwd_3 / fwd_5; "Mamba-2 offers a different
 * scaling path": chunk_cumsum, fwd_pass_state, compute_out).  The backward
 * returns the gradients of L = <dy, y> + <dfinal, final> with respect to every
 * input (same kernel table, bwd_5 .. bwd_16; the forward states are recomputed
 * inside ssd_bwd, as bwd_5 and bwd_6 do on the pages).
 *
 * Conventions shared by every entry point
 *   - All tensors are dense, row-major, caller-owned DEVICE memory on the
 *     current CUDA device.  The library never allocates, frees or keeps a
 *     pointer after the call returns (asynchronously, on `stream`).
 *   - Shapes (B = batch, T = seqlen, H = nheads, P = headdim, N = dstate,
 *     G = ngroups):
 *         x, y, dy, dx         (B, T, H, P)     dtype in_dtype / out_dtype / in_dtype / f32
 *         dt, ddt              (B, T, H)        in_dtype / f32
 *         B, C, dB, dC         (B, T, G, N)     in_dtype / f32
 *         dt_bias, A, D, dA, dD, ddt_bias   (H) f32
 *         init, final, dfinal, dinit        (B, H, P, N) f32
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     launch goes to that stream; no call synchronises the host.
 *   - Every pointer must be aligned to its element size; the tensor-core fast
 *     path additionally needs 16-byte alignment of x, B, C, dy, y (it is only
 *     chosen when that holds).
 *   - Errors: a host-side check that fails returns before anything is
 *     launched.  A failed launch returns SSD_ERR_CUDA.  Kernels never trap:
 *     a bounded wait that times out on the device records SSD_ERR_TIMEOUT in a
 *     device status word, which ssd_get_device_status() reads and clears.
 *   - No entry point throws or exits; all are thread-safe.
 */
#ifndef SSD_H_
#define SSD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1, /* bad shape, NULL required pointer, misalignment */
  SSD_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement   */
  SSD_ERR_WORKSPACE = 3,   /* workspace NULL or smaller than the size query   */
  SSD_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed            */
  SSD_ERR_TIMEOUT = 5,     /* a device-side bounded wait expired              */
  SSD_ERR_NONFINITE = 6    /* an output holds NaN or Inf (opt-in check)       */
} ssd_status;

/* Bytes of the fixed scratch array behind ssd_fwd_noalloc (64 MiB). */
#define SSD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

/* Problem description.  Limits: every extent >= 1; nheads % ngroups == 0;
 * 1 <= chunk_size <= 256; headdim * dstate <= 16384.  seqlen need not be a
 * multiple of chunk_size (the last chunk is partial). */
typedef struct {
  int64_t batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size;
  int32_t in_dtype;  /* ssd_dtype of x, dt, B, C (and dy in ssd_bwd) */
  int32_t out_dtype; /* ssd_dtype of y                                */
} ssd_shape;

/* Byte offsets, inside the ssd_fwd workspace, of the intermediates the
 * forward leaves there (all f32; nc = ceil(seqlen / chunk_size)):
 *   delta     (B, H, nc, L)       softplus(dt + dt_bias), 0 on the padded tail
 *   dA_cumsum (B, H, nc, L)       in-chunk inclusive cumsum of delta * A
 *   states    (B, nc, H, P, N)    chunk_state output S_c
 *   hprev     (B, nc, H, P, N)    state entering chunk c (state_passing output)
 * They stay valid until the workspace is reused.  When the call took the
 * tensor-core path (ssd_last_path() == 1), the hprev bytes hold each state
 * split into bf16 hi = rn(v) and lo = rn(v - hi) in the kernels'
 * shared-memory layout instead of f32: per (b, c, h) and 64-row half of the
 * state (one half at headdim 64, rows 0-63 then 64-127 at headdim 128) N/64
 * "hi" panels then N/64 "lo" panels, each 64 rows of 128 bytes (64 bf16 of
 * one row p); the 16-byte chunk j of row p is stored at chunk j ^ (p % 8). */
typedef struct {
  size_t delta, dA_cumsum, states, hprev, total;
} ssd_fwd_layout;

/* Workspace bytes needed by ssd_fwd / ssd_bwd for this shape (0 if the shape
 * is invalid).  The workspace is caller-owned device memory, 256-byte aligned. */
size_t ssd_fwd_workspace_size(const ssd_shape* shape);
size_t ssd_bwd_workspace_size(const ssd_shape* shape);
int ssd_fwd_workspace_layout(const ssd_shape* shape, ssd_fwd_layout* out);

/* Forward.  dt_bias, D, init and final_states may be NULL (zero bias, no skip
 * term, zero initial state, final state not written). */
int ssd_fwd(const ssd_shape* shape, const void* x, const void* dt, const float* dt_bias,
            const float* A, const void* B, const void* C, const float* D,
            const float* init_states, void* y, float* final_states, void* workspace,
            size_t workspace_bytes, void* stream);

/* Backward.  Takes the forward inputs (not saved states) plus dy and an
 * optional dfinal_states (NULL = 0).  Writes dx, ddt (w.r.t. the raw dt
 * input), dA, dB and dC (summed over the heads of each group); dD, ddt_bias
 * and dinit_states may be NULL (not written).  Reductions are deterministic:
 * repeated calls give bit-identical results. */
int ssd_bwd(const ssd_shape* shape, const void* x, const void* dt, const float* dt_bias,
            const float* A, const void* B, const void* C, const float* D,
            const float* init_states, const void* dy, const float* dfinal_states, float* dx,
            float* ddt, float* dA, float* dB, float* dC, float* dD, float* ddt_bias,
            float* dinit_states, void* workspace, size_t workspace_bytes, void* stream);

/* Synchronises `stream`, returns the device status word of the current
 * device (SSD_OK, SSD_ERR_TIMEOUT or SSD_ERR_NONFINITE) and clears it.  The
 * outputs of a call are only meaningful once this word reads SSD_OK: a
 * kernel whose bounded wait expired skips the rest of its work. */
int ssd_get_device_status(void* stream);

/* Opt-in scan of every output for NaN / Inf ("End-to-end validation": no NaNs
 * and no loss spikes).  With enable != 0, each later ssd_fwd, ssd_fwd_noalloc
 * and ssd_bwd launches, after its kernels and on the same stream, one more
 * kernel that reads every output it wrote (y, final_states; dx, ddt, dA, dB,
 * dC and, when requested, dD, ddt_bias, dinit_states) and records
 * SSD_ERR_NONFINITE in the device status word if any element is NaN or Inf
 * (an earlier SSD_ERR_TIMEOUT is kept).  Read it with ssd_get_device_status.
 * The scan reads the outputs once more (bandwidth-bound).  Process-wide;
 * returns the previous setting.  Default: off. */
int ssd_set_check_finite(int enable);

/* Which kernel family the last ssd_fwd / ssd_bwd on this host thread used:
 * 0 = generic SIMT path, 1 = tcgen05 tensor-core path.  The tensor-core path
 * takes bf16 inputs with headdim 64 or 128, dstate 64 or 128, chunk_size 128
 * or 256, x / B / C / y / dy / dx / dB / dC / states 16-byte aligned, and an
 * even nheads / ngroups at headdim 64; everything else runs on the generic
 * kernels. */
int ssd_last_path(void);

/* Optional per-kernel timing.  ssd_profile_enable(1) clears the counters and
 * brackets every later kernel launch of this library with two CUDA events on
 * its launch stream; ssd_profile_enable(0) stops.  ssd_profile_read waits for
 * the recorded events and writes, for up to max_kernels kernel names, the name
 * (64 bytes each, NUL-terminated, into `names`), the summed device time in ms
 * and the number of launches; it returns the number of entries (or
 * -SSD_ERR_CUDA).  Any output pointer may be NULL. */
int ssd_profile_enable(int on);
int ssd_profile_read(int max_kernels, char* names, double* ms, int64_t* launches);

/* Number of kernels this library has launched in this process. */
int64_t ssd_launch_count(void);

/* Forward pass for callers that cannot allocate device memory (no workspace
 * argument).  The pages have no counterpart: this is a convenience of this
 * library.  Callers such as a host runtime whose memory pool already owns the
 * device, a plugin that is handed only its tensors, or a latency-critical loop
 * that cannot afford cudaMalloc (which may synchronise the device) use it
 * instead of ssd_fwd.
 *   - Scratch: a fixed array of SSD_NOALLOC_SCRATCH_BYTES (64 MiB; also
 *     ssd_noalloc_scratch_bytes()) of device memory inside the library, held
 *     on every GPU that loads the library until the process exits.  Shapes
 *     whose ssd_fwd_workspace_size() exceeds it return SSD_ERR_WORKSPACE;
 *     nothing is launched.
 *   - The scratch used is the one of the CURRENT device (cudaGetDevice), like
 *     every other pointer argument: `stream` must belong to that device.
 *   - Inputs, outputs, results and errors are those of ssd_fwd.  It calls no
 *     cudaMalloc, cudaFree or other allocating routine.
 *   - The first call on each device (and the first after the device's
 *     context changed, e.g. after cudaDeviceReset or under another driver
 *     context) looks up the scratch's device address with that device
 *     current and caches it with the context; make that first call before
 *     any stream capture.
 *   - Every call on a device shares the one scratch array and leaves the last
 *     call's intermediates in it: calls that overlap on the GPU (different
 *     streams, or host threads without ordering between them) race and give
 *     wrong results.  Order them, e.g. on one stream. */
int ssd_fwd_noalloc(const ssd_shape* shape, const void* x, const void* dt, const float* dt_bias,
                    const float* A, const void* B, const void* C, const float* D,
                    const float* init_states, void* y, float* final_states, void* stream);
size_t ssd_noalloc_scratch_bytes(void);

/* Context (sequence) parallelism.  With the sequence split into contiguous
 * segments r = 0 .. R-1, one per rank, the recurrence maps a segment's
 * incoming state affinely, H_out(r) = D_r * H_in(r) + F_r, where F_r is the
 * segment's final state from a zero initial state and D_r its total decay
 * (the recurrence of "Mamba-2 offers a different scaling path", taken over
 * the whole segment; the pages name sequence sharding as future work in
 * "Closing thoughts").  Rank r's incoming state is an exclusive scan of these
 * maps over the ranks before it; the gradient of its outgoing state is the
 * same scan over the ranks after it, applied to the initial-state gradients.
 *
 * ssd_segment_decay: decay[b, h] = exp(A[h] * sum_t softplus(dt[b,t,h] +
 * dt_bias[h])) over the shape's seqlen (the sum in fp64, split over the
 * sequence and added back in a fixed order).  Uses shape->batch, seqlen,
 * nheads and in_dtype (dt's dtype); dt (B, T, H), dt_bias (H) or NULL, A
 * (H), decay (B, H) f32, device memory; workspace of
 * ssd_segment_decay_workspace_size(shape) bytes (8-byte aligned,
 * caller-owned; the size depends on the current device's SM count).
 * Asynchronous on `stream`.  Returns SSD_ERR_INVALID_ARG for a NULL
 * required pointer or a bad shape (seqlen must be below 2^30),
 * SSD_ERR_WORKSPACE for a missing or small workspace. */
size_t ssd_segment_decay_workspace_size(const ssd_shape* shape);
int ssd_segment_decay(const ssd_shape* shape, const void* dt, const float* dt_bias,
                      const float* A, float* decay, void* workspace, size_t workspace_bytes,
                      void* stream);

/* ssd_state_scan: out = the exclusive scan of the maps S -> D_k * S + S_k
 * for rank `rank` of `nranks`: direction 0 runs over k = 0 .. rank-1
 * (incoming state; S_0 is rank 0's final state with its own initial state),
 * direction 1 over k = nranks-1 .. rank+1 (gradient of the outgoing state;
 * S_{R-1} is the last rank's initial-state gradient with the caller's
 * final-state gradient).  decays (nranks, bh) f32, states (nranks, bh, pn)
 * f32, out (bh, pn) f32, device memory; bh = batch * nheads, pn = headdim *
 * dstate.  Asynchronous on `stream`.  Returns SSD_ERR_INVALID_ARG for a rank
 * outside [0, nranks), a direction other than 0 / 1, empty sizes or a NULL
 * pointer. */
int ssd_state_scan(int nranks, int rank, int direction, int64_t bh, int64_t pn,
                   const float* decays, const float* states, float* out, void* stream);

/* ssd_fwd_final_state: the final state only, H_out = the state after the
 * shape's seqlen from init_states (NULL: zero): chunk_cumsum, chunk_state
 * and state_passing of ssd_fwd without chunk_scan (C and D are not read).
 * Arguments as for ssd_fwd; final_states (B, H, P, N) f32.  Workspace: at
 * least ssd_fwd_workspace_size(shape) bytes, 256-byte aligned, caller-owned.
 * Asynchronous on `stream`.  Errors as ssd_fwd. */
int ssd_fwd_final_state(const ssd_shape* shape, const void* x, const void* dt,
                        const float* dt_bias, const float* A, const void* B,
                        const float* init_states, float* final_states, void* workspace,
                        size_t workspace_bytes, void* stream);

/* ssd_bwd_dinit: the gradient of <dy, y> + <dfinal, final> with respect to
 * the initial state only: dinit = G_0 of the reverse chunk recurrence
 * G_c = dH^scan_c + exp(a_c[L-1]) G_{c+1}, G_nc = dfinal_states (NULL:
 * zero), with dH^scan_c = sum_l exp(a_l) dy_l (x) C_l.  It depends on dt,
 * dt_bias, A, C and dy only (x and B are not read).  dt (B, T, H), C
 * (B, T, G, N), dy (B, T, H, P) in shape->in_dtype; dt_bias (H) or NULL, A
 * (H), dfinal_states and dinit_states (B, H, P, N) f32.  Workspace: at least
 * ssd_fwd_workspace_size(shape) bytes, 256-byte aligned, caller-owned.
 * Asynchronous on `stream`.  Errors as ssd_bwd. */
int ssd_bwd_dinit(const ssd_shape* shape, const void* dt, const float* dt_bias, const float* A,
                  const void* C, const void* dy, const float* dfinal_states,
                  float* dinit_states, void* workspace, size_t workspace_bytes, void* stream);

/* Gated RMSNorm: the normalisation that follows the SSD output in a Mamba-2
 * layer; its backward is the pages' _layer_norm_bwd (step bwd_2 of the
 * per-kernel table in "Latency and speedup by kernel").  The pages name the
 * kernel but not its arithmetic; the reading implemented is the layer's
 * output norm with the gate before the norm: with u = y * silu(z), per row
 * and group g of group_size consecutive features,
 *     rstd_g = 1 / sqrt(mean_g(u^2) + eps),   out = u * rstd_g * w,
 * and the backward of <dout, out> with respect to y, z and w.  Rows are the
 * (batch * seqlen) positions, features the (nheads * headdim) channels.
 * Requirements: rows < 2^30, features and group_size multiples of 8,
 * group_size dividing features (else SSD_ERR_INVALID_ARG); features <= 4096,
 * features / 8 a multiple of 32 or a power of two below 32, group_size / 8 a
 * multiple of 32 or a power of two below 32 (else SSD_ERR_UNSUPPORTED).
 * Kernels: rows stream through shared memory by bulk asynchronous copies;
 * waits are bounded (1 s) and an expired wait records SSD_ERR_TIMEOUT in
 * the device status word (ssd_get_device_status). */
typedef struct {
  int64_t rows, features, group_size;
  float eps;
  int32_t in_dtype;  /* ssd_dtype of y, z and dout  */
  int32_t out_dtype; /* ssd_dtype of out, dy and dz */
} ssd_norm_shape;

/* Bytes of workspace ssd_gated_norm_bwd needs (per-CTA partial sums of dw);
 * 0 for an invalid or unsupported shape.  Depends on the current device's SM
 * count. */
size_t ssd_gated_norm_workspace_size(const ssd_norm_shape* shape);

/* ssd_gated_norm_fwd: y, z (rows, features) in_dtype, w (features) f32,
 * out (rows, features) out_dtype; rstd (rows, features / group_size) f32 or
 * NULL (saved for the backward).  y, z, out 16-byte aligned; device memory;
 * asynchronous on `stream`.  rows == 0 launches nothing.  Errors:
 * SSD_ERR_INVALID_ARG (shape, NULL or misaligned pointer),
 * SSD_ERR_UNSUPPORTED, SSD_ERR_CUDA. */
int ssd_gated_norm_fwd(const ssd_norm_shape* shape, const void* y, const void* z,
                       const float* w, void* out, float* rstd, void* stream);

/* ssd_gated_norm_bwd: gradients of <dout, out>: dy, dz (rows, features)
 * out_dtype, dw (features) f32 (the sum over rows, taken in a fixed order).
 * rstd as ssd_gated_norm_fwd wrote it, or NULL to recompute it.  y, z, dout,
 * dy, dz 16-byte aligned; workspace of ssd_gated_norm_workspace_size bytes,
 * 16-byte aligned, caller-owned.  rows == 0 sets dw to 0.  Errors as
 * ssd_gated_norm_fwd, plus SSD_ERR_WORKSPACE. */
int ssd_gated_norm_bwd(const ssd_norm_shape* shape, const void* y, const void* z,
                       const float* w, const float* rstd, const void* dout, void* dy, void* dz,
                       float* dw, void* workspace, size_t workspace_bytes, void* stream);

/* Launch configuration of the gated-norm kernels for one shape, as an
 * offline sweep chooses it (the pages' ahead-of-time config generator,
 * "Cutting autotuning overhead with an automated config generator", Fig. 4:
 * search per environment ahead of time, store the result, load it at start):
 * rows_per_item = rows per CTA work
 * item (the CTA has rows_per_item * features / 8 threads, at most 512 and a
 * multiple of 32; it applies to the backward, and to the forward where that
 * keeps one 8-feature vector per thread: a forward with two vectors per
 * thread takes as many rows as fill 512 threads); ring_kb = shared-memory ring size aimed at per CTA
 * (8 .. 200); ctas_per_sm = persistent CTAs per SM at most (1 .. 8).  A zero
 * field keeps the built-in choice. */
typedef struct {
  int32_t rows_per_item, ring_kb, ctas_per_sm;
} ssd_norm_config;

/* Sets (config != NULL) or removes (NULL) the table entry for shape's
 * (features, group_size, in_dtype, out_dtype); rows and eps are ignored.
 * Thread-safe; at most 64 entries (else SSD_ERR_UNSUPPORTED).  Returns
 * SSD_ERR_INVALID_ARG for an invalid shape or field. */
int ssd_gated_norm_set_config(const ssd_norm_shape* shape, const ssd_norm_config* config);

/* The configuration the next call with this shape will use (the table's
 * fields where set, the built-in choice elsewhere) in *out.  Returns 1 if a
 * table entry exists, 0 if not, -SSD_ERR_INVALID_ARG for a bad shape. */
int ssd_gated_norm_get_config(const ssd_norm_shape* shape, ssd_norm_config* out);

/* Launch table of the SSD chunk kernels (the tensor-core path), the SSD side
 * of the offline config generator of "Cutting autotuning overhead with an
 * automated config generator" (Fig. 4): a sweep finds the best launch per
 * shape ahead of time, and the table is applied when the library loads.
 * Each kernel's CTAs cover (batch, chunk, 128-row tile, group, block of
 * heads); with chunk 256 a chunk has two row tiles, one with twice the
 * column panels of the other (the heavy tile, launched first).
 *   scan_head_blocks: the blocks chunk_scan splits a group's heads into for
 *     the heavy tile, scan_head_blocks_light for the other;
 *   bc_head_blocks, bc_head_blocks_light: the same for the dC and dB
 *     kernels, whose per-block partial sums live in the ssd_bwd workspace
 *     (so they change ssd_bwd_workspace_size: query the size after setting
 *     the table).
 * With chunk 128 (one row tile) the light fields are ignored.  0 keeps the
 * built-in rule's count (a list-scheduling model of the launch); a nonzero
 * value must divide the heads per group and be at most 32.  The kernels see
 * a head of headdim 128 as two 64-wide heads, so there the blocks split
 * 2 * nheads / ngroups heads. */
typedef struct {
  int32_t scan_head_blocks, bc_head_blocks;
  int32_t scan_head_blocks_light, bc_head_blocks_light;
} ssd_scan_config;

/* Sets (config != NULL) or removes (NULL) the entry of shape's (batch,
 * seqlen, nheads, headdim, dstate, ngroups, chunk_size).  Thread-safe; at
 * most 64 entries (else SSD_ERR_UNSUPPORTED); SSD_ERR_INVALID_ARG for an
 * invalid shape or field. */
int ssd_scan_set_config(const ssd_shape* shape, const ssd_scan_config* config);

/* The head blocks the next ssd_fwd / ssd_bwd with this shape will use (the
 * table's where set, the built-in rule's elsewhere) in *out.  Returns 1 if a
 * table entry exists, 0 if not, -SSD_ERR_INVALID_ARG for a bad shape. */
int ssd_scan_get_config(const ssd_shape* shape, ssd_scan_config* out);

/* Diagnostic: one tcgen05 tile product on the current device,
 * D[128][nn] = A[128][k] * B[nn][k]^T (A, B bf16 row-major, D f32 row-major,
 * all device memory), with A and B staged in shared memory K-major (0) or
 * MN-major (1) in the 128-byte-swizzle layout of the tensor-core kernels;
 * swap_mn_offsets exchanges the two byte offsets of MN-major descriptors.
 * 16 <= nn <= 256, nn % 16 == 0 (nn % 64 == 0 when b_mn); 16 <= k <= 128,
 * k % 16 == 0; A and B 16-byte aligned.  Asynchronous on `stream`. */
int ssd_selftest_mma(int a_mn, int b_mn, int swap_mn_offsets, int nn, int k, const void* A,
                     const void* B, float* D, void* stream);

/* Diagnostic: launches one kernel whose only work is a wait on a barrier
 * that nothing completes.  The library's bounded wait gives up after about one
 * second, records SSD_ERR_TIMEOUT in the device status word and the kernel
 * returns; the CUDA context stays usable.  Lets callers check their handling
 * of ssd_get_device_status() without any GPU fault.  Asynchronous. */
int ssd_selftest_timeout(void* stream);

/* Diagnostic: as ssd_selftest_timeout, with the suspending bounded wait
 * (mbarrier try_wait with a suspend-time hint) that the gated-norm kernels'
 * row ring uses; it too records SSD_ERR_TIMEOUT after about 1 s and returns. */
int ssd_selftest_timeout_suspend(void* stream);

/* Static description of a status code. */
const char* ssd_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* SSD_H_ */
