/*
 * kda.h -- C ABI of libkda, a GB300 (sm_103a) implementation of the chunked
 * Kimi Delta Attention (KDA) forward pass and its backward.
 *
 * The operation (page "feat(kda): integrate KDA attention with tokamax backend
 * and CP support", section "Delta Rule formulation"), per batch row b and head
 * h, token by token, with a K x V state S indexed [key][value]:
 *
 *     S'       = S * exp(g_t)        g_t in R^K: per-key-channel log-decay
 *     residual = v_t - k_t^T S'
 *     S        = S' + beta_t * k_t (outer) residual
 *     o_t      = scale * q_t^T S
 *
 * computed in chunks of 64 tokens (same page, section "Public API":
 * chunk_kda(..., chunk_size=64, initial_state, output_final_state,
 * segment_ids, ...)).  Packed variable-length sequences are given by 1-based
 * segment ids [B, T] with 0 = padding (same section, decoder_segment_ids);
 * the state restarts at every segment boundary.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers to contiguous row-major
 *     buffers owned by the caller.  libkda allocates no device memory and
 *     keeps no global state between calls (the status word lives in the
 *     caller's workspace), so calls are reentrant; calls on different
 *     streams must use different workspaces.
 *   - Work is enqueued on `stream` and the call returns without
 *     synchronising.  Argument errors are detected on the host before
 *     anything is enqueued and are returned synchronously; nothing is
 *     thrown across the ABI.
 *   - Device-side conditions (a bounded wait that ran out, a debug-mode
 *     bounds check) set bits in the status word at the start of the
 *     workspace; read them with kda_read_device_status() after the work has
 *     finished.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_VERSION 100 /* 1.0.0 */

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st *kda_stream_t;

typedef enum kda_status {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,  /* NULL required pointer, bad size, bad flag   */
  KDA_ERR_UNSUPPORTED = 2,  /* shape / dtype / chunk size not implemented   */
  KDA_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned             */
  KDA_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than required      */
  KDA_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed         */
  KDA_ERR_TIMEOUT = 6,      /* device status: a bounded wait ran out        */
  KDA_ERR_DEVICE = 7        /* device status: another device-side error     */
} kda_status;

typedef enum kda_dtype {
  KDA_DTYPE_F32 = 0,
  KDA_DTYPE_BF16 = 1
} kda_dtype;

/* Problem shape.  q, k: [B,T,H,K]; v, o: [B,T,H,V], all of qkv_dtype.
 * g: [B,T,H,K] float32; beta: [B,T,H] float32; states [B,H,K,V] float32.
 * Supported: K, V in {32, 64, 128}; B, T, H >= 1; B*T*H*max(K,V) < 2^31. */
typedef struct kda_shape {
  int B, T, H, K, V;
  kda_dtype qkv_dtype;
} kda_shape;

/* Implementation choice for kda_chunk_fwd_ex. */
typedef enum kda_impl {
  KDA_IMPL_AUTO = 0,  /* fastest that applies: SPLIT when the workspace is
                         large enough, else TC, else SIMT.  With segment
                         ids and the split path it always computes the
                         result: runs that overflow the split workspace are
                         served by the fused TC kernel on the device.
                         Without segment ids, when at least 3 segments fill
                         the SMs (few rows x heads) and each holds 8 or
                         more chunks (32 or more when there are fewer than
                         8 segments), and the workspace holds the scan's
                         buffers, SPLIT runs as the chunk-parallel scan of
                         kda_chunk_fwd_scan.                                */
  KDA_IMPL_SIMT = 1,  /* fp32 CUDA-core kernel (every supported shape)      */
  KDA_IMPL_TC = 2,    /* fused tcgen05 / TMA kernel: bf16, K = V = 128      */
  KDA_IMPL_SPLIT = 3  /* tcgen05 in two kernels (parallel per-chunk prep,
                         then the state recurrence): bf16, K = V = 128,
                         value tile 32 or 64 (v_tile 0: 32 when every
                         (row, head, tile) fits one CTA per SM and there are
                         no segment ids, else 64); needs the larger
                         workspace reported by
                         kda_chunk_fwd_workspace_size_for(.., KDA_IMPL_SPLIT) */
} kda_impl;

/* Device status bits OR-ed into the workspace status word. */
#define KDA_DEVICE_TIMEOUT 0x1u    /* a bounded mbarrier / flag wait ran out */
#define KDA_DEVICE_BAD_INPUT 0x2u  /* a debug-build input check failed       */
#define KDA_DEVICE_WORKSPACE 0x4u  /* the runs need more chunk items than the
                                      workspace was sized for (split path) */

/*
 * Bytes of workspace that let kda_chunk_fwd run its fastest kernel on this
 * shape (the same as kda_chunk_fwd_workspace_size_for(s, has_segment_ids,
 * KDA_IMPL_AUTO)).  The workspace holds the device status word, when
 * segment ids are given the run list (one 8-byte record per run, at most
 * B*T runs) and per-row counts, and for the tensor-core split path the
 * per-chunk operands.  Any smaller workspace of at least
 * kda_chunk_fwd_workspace_size_for(s, has_segment_ids, KDA_IMPL_SIMT) bytes
 * is accepted too; AUTO then picks a kernel that fits it, which can be
 * several times slower.  The workspace must be zero-filled once before its
 * first use (for instance allocated with cudaMemset 0); libkda leaves it
 * reusable.  Returns 0 when `s` is NULL or invalid.
 */
KDA_API size_t kda_chunk_fwd_workspace_size(const kda_shape *s, int has_segment_ids);

/*
 * Workspace bytes implementation `impl` needs (same zero-fill rule).  For
 * KDA_IMPL_SPLIT this holds the per-chunk operands the recurrence kernel
 * reads: about 73 KB per (row, 64-token chunk, head).  With segment ids the
 * chunks are those of each run, so their number depends on the runs: the
 * size returned here assumes at most ceil(T/64) runs per row (see
 * kda_chunk_fwd_workspace_size_packed for another bound).  For
 * KDA_IMPL_AUTO it is the size that lets AUTO pick its fastest kernel.
 * Returns 0 when the shape or the choice is invalid or does not apply.
 */
KDA_API size_t kda_chunk_fwd_workspace_size_for(const kda_shape *s,
                                                int has_segment_ids,
                                                kda_impl impl);

/*
 * Split-path workspace for packed inputs with at most max_runs_per_row runs
 * in any row (the pages' bound on segments per row, max_segments_per_seq):
 * room for B * (ceil(T/64) + max_runs_per_row) chunk items.  When the runs
 * of a call need more chunk items than its workspace holds, the split path
 * computes nothing and sets KDA_DEVICE_WORKSPACE in the status word
 * (kda_read_device_status then returns KDA_ERR_WORKSPACE).  Returns 0 for an
 * invalid shape, a shape the split path does not serve, or a bound < 1.
 */
KDA_API size_t kda_chunk_fwd_workspace_size_packed(const kda_shape *s,
                                                   int max_runs_per_row);

/*
 * Chunked KDA forward (the operation above).
 *   q, k, v       device, [B,T,H,K|V] of s->qkv_dtype, 16-byte aligned.
 *   g             device float32 [B,T,H,K]: log-decay, already activated
 *                 (use_gate_in_kernel=False on the pages).  Contract:
 *                 g in [-5, 0] (the pages' safe-gate lower bound range);
 *                 values below -5 may lose accuracy in the intra-chunk
 *                 factors, values above 0 are growth and are not supported.
 *   beta          device float32 [B,T,H].
 *   scale         output scale (the pages leave its default open; callers
 *                 usually pass K^-0.5).
 *   chunk_size    must be 64.
 *   initial_state device float32 [B,H,K,V] or NULL (zeros).  It seeds only
 *                 the first run of each row; later runs start from zero.
 *   segment_ids   device int32 [B,T], 1-based ids, 0 = padding, or NULL
 *                 (every token has id 1).  A run is a maximal span of equal
 *                 non-zero ids; padding tokens get o = 0, do not touch the
 *                 state and end the current run.
 *   o             device [B,T,H,V] of s->qkv_dtype (written for every token).
 *   final_state   device float32 [B,H,K,V] or NULL (not requested): the state
 *                 after each row's last non-padding token (initial_state or
 *                 zeros for an all-padding row).
 *   workspace     device, 256-byte aligned, zero-filled before first use;
 *                 kda_chunk_fwd_workspace_size(s, segment_ids != NULL) bytes
 *                 for the fastest kernel, at least the KDA_IMPL_SIMT size of
 *                 kda_chunk_fwd_workspace_size_for (KDA_ERR_WORKSPACE when
 *                 smaller).
 * Returns KDA_OK or an error code; on error nothing has been enqueued.
 */
KDA_API kda_status kda_chunk_fwd(const kda_shape *s, const void *q, const void *k,
                         const void *v, const float *g, const float *beta,
                         float scale, int chunk_size,
                         const float *initial_state,
                         const int32_t *segment_ids, void *o,
                         float *final_state, void *workspace,
                         size_t workspace_bytes, kda_stream_t stream);

/*
 * Same as kda_chunk_fwd with an explicit implementation and value-tile
 * width (v_tile = columns of V one CTA owns; 0 = automatic; otherwise a
 * divisor of V supported by the chosen kernel).  KDA_ERR_UNSUPPORTED when
 * the choice does not apply to the shape.
 */
KDA_API kda_status kda_chunk_fwd_ex(const kda_shape *s, const void *q, const void *k,
                            const void *v, const float *g, const float *beta,
                            float scale, int chunk_size,
                            const float *initial_state,
                            const int32_t *segment_ids, void *o,
                            float *final_state, void *workspace,
                            size_t workspace_bytes, kda_impl impl, int v_tile,
                            kda_stream_t stream);

/*
 * The chunked forward computed as a chunk-parallel state scan, for rows
 * without segment ids (the single-GPU counterpart of the state chain of the
 * pages' context parallelism: page "feat(kda): integrate KDA attention with
 * tokamax backend and CP support", section "Implementation Details").  Each
 * row's 64-token chunks are cut into n_segments contiguous segments.  The
 * chunk form is affine in the state entering a chunk, so each segment but
 * the last maps its entering state S to M S + B (M: K x K, B: K x V, both
 * computed in parallel over segments, rows and heads), the segments'
 * entering states are chained from initial_state in fp32, and then every
 * segment's chunks run in parallel from their entering state.  It trades
 * about three times the state-recurrence work for a chain n_segments times
 * shorter, which pays when few (row, head) pairs leave SMs idle and T is
 * long.  Arguments, layouts and results are those of kda_chunk_fwd with
 * segment_ids = NULL (up to rounding: the maps are rounded like the state).
 *   n_segments  0 (choose: as many segments as the final pass's units of
 *               64 state columns fit the GPU's SMs, i.e. SMs / (2 B H), at
 *               least 2) or >= 2; capped at ceil(T/64) and
 *               rounded so every segment holds at least one chunk.
 *   workspace   device, kda_chunk_fwd_scan_workspace_size(s, n_segments)
 *               bytes, 256-byte aligned, zero-filled before first use.
 * bf16 q/k/v with K = V = 128 and T > 64 only (KDA_ERR_UNSUPPORTED
 * otherwise; the workspace query then returns 0); KDA_ERR_INVALID_ARG for
 * n_segments < 0 or == 1.  Asynchronous on `stream`.
 */
KDA_API size_t kda_chunk_fwd_scan_workspace_size(const kda_shape *s, int n_segments);
/* The segment count kda_chunk_fwd_scan uses for this request (0 when the
 * shape or the request is not served). */
KDA_API int kda_chunk_fwd_scan_segments(const kda_shape *s, int n_segments);
KDA_API kda_status kda_chunk_fwd_scan(const kda_shape *s, const void *q, const void *k,
                                      const void *v, const float *g, const float *beta,
                                      float scale, int chunk_size, const float *initial_state,
                                      void *o, float *final_state, int n_segments,
                                      void *workspace, size_t workspace_bytes,
                                      kda_stream_t stream);

/*
 * kda_chunk_fwd without a workspace argument, for callers that cannot
 * allocate device memory (no counterpart on the pages: it exists only for
 * such callers).  A plugin inside a host application may be handed nothing
 * but the tensors it works on; other code runs under a memory budget held
 * by another allocator, or on a path where allocating is not allowed.  The
 * arguments and results are those of kda_chunk_fwd.  The scratch it needs
 * lives in a fixed device array of KDA_NOALLOC_SCRATCH_BYTES bytes that the
 * library defines; every GPU that loads the library keeps that memory until
 * the process exits.  The call itself allocates nothing.
 *   - Argument errors are the codes kda_chunk_fwd returns for the same
 *     input.  Shapes whose smallest workspace,
 *     kda_chunk_fwd_workspace_size_for(s, segment_ids != NULL,
 *     KDA_IMPL_SIMT), exceeds KDA_NOALLOC_SCRATCH_BYTES are rejected with
 *     KDA_ERR_WORKSPACE (with segment ids about B*T > 130000 tokens).  The
 *     kernel is the one AUTO picks for a workspace of that many bytes.
 *   - All calls share the array: calls whose work overlaps on the GPU race
 *     and give wrong results.  Order them on one stream.
 *   - The array's address is looked up on the first call in each CUDA
 *     context of a device, with that device current, and kept for that
 *     context; after a device reset the next call looks it up again.  Make
 *     the first call on a device before any stream capture begins.
 *   - Each call clears the array's header on `stream` before its kernels,
 *     so the previous call's counters never carry over; the device status
 *     bits of the last call stay there until the next call, and
 *     kda_chunk_fwd_noalloc_status reads them.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (1u << 20)
KDA_API kda_status kda_chunk_fwd_noalloc(
    const kda_shape *s, const void *q, const void *k, const void *v,
    const float *g, const float *beta, float scale, int chunk_size,
    const float *initial_state, const int32_t *segment_ids, void *o,
    float *final_state, kda_stream_t stream);

/*
 * Device status of the last kda_chunk_fwd_noalloc call on the current
 * device (no counterpart on the pages): waits for `stream`, then reads the
 * status word of the fixed scratch array into *device_bits, with the
 * return codes of kda_read_device_status.  KDA_ERR_INVALID_ARG for a NULL
 * device_bits.
 */
KDA_API kda_status kda_chunk_fwd_noalloc_status(kda_stream_t stream, uint32_t *device_bits);

/*
 * 1 when `impl` can run shape `s` (KDA_IMPL_AUTO: always, for a valid
 * shape), else 0.  Pure host query.
 */
KDA_API int kda_impl_available(kda_impl impl, const kda_shape *s, int v_tile);

/*
 * Short-convolution prologue (page "feat(kda): ...", section "Layer
 * architecture", step 1: causal depthwise 1-D conv of width 4 with SiLU on
 * each of Q, K, V; optional step 5 / use_qk_l2norm_in_kernel: L2 norm of q
 * and k per token and head).  Per channel c of each input:
 *     y_t[c] = SiLU( sum_{i=0}^{3} w[c][3-i] * x_{t-i}[c] )
 * with taps before t = 0 or before the start of t's run equal to zero, no
 * bias, and y = 0 on padding tokens.  With l2norm_qk != 0, q and k are then
 * scaled per (token, head) by 1 / sqrt(sum y^2 + 1e-6).  fp32 arithmetic;
 * the sigmoid uses the approximate exp2 and reciprocal instructions
 * (relative error a few fp32 ulp); bf16 outputs are rounded to nearest.
 *   x_q, x_k      device [B,T,H,K] of s->qkv_dtype; x_v [B,T,H,V].
 *   w             device float32, three weight blocks back to back:
 *                 w_q [H*K][4], w_k [H*K][4], w_v [H*V][4].
 *   segment_ids   device int32 [B,T] or NULL.
 *   q, k, v       device outputs, same shapes and dtype as the inputs; they
 *                 must not alias the inputs.
 * Every pointer must be 16-byte aligned (KDA_ERR_ALIGNMENT).  Returns
 * KDA_ERR_UNSUPPORTED when B * ceil(T / 24) exceeds 65535; the call is
 * asynchronous on `stream`.
 */
KDA_API kda_status kda_short_conv_silu(const kda_shape *s, const void *x_q,
                               const void *x_k, const void *x_v,
                               const float *w, const int32_t *segment_ids,
                               int l2norm_qk, void *q, void *k, void *v,
                               kda_stream_t stream);

/*
 * Waits for `stream`, then reads the device status word at the start of
 * `workspace` into *device_bits (KDA_DEVICE_* bits, 0 when clean).  Returns
 * KDA_ERR_TIMEOUT when the timeout bit is set, KDA_ERR_WORKSPACE for the
 * workspace bit, KDA_ERR_DEVICE for any other bit, KDA_OK when clean,
 * KDA_ERR_CUDA when the copy fails.
 */
KDA_API kda_status kda_read_device_status(const void *workspace, kda_stream_t stream,
                                  uint32_t *device_bits);

/* Enqueues a reset of the device status word to zero on `stream`. */
KDA_API kda_status kda_clear_device_status(void *workspace, kda_stream_t stream);

/*
 * End to end on HOST buffers (an API shape of this library, not of the
 * pages): q, k, v, g, beta, initial_state, segment_ids, o and final_state
 * are host pointers in the layouts of kda_chunk_fwd (pin them with
 * cudaHostAlloc or cudaHostRegister, else the copies are synchronous).
 * The call copies the inputs in, runs the forward and copies o and
 * final_state back, with the copies overlapped with the compute.  Without
 * segment ids it pipelines over time: the tokens are split into ranges of
 * a multiple of 64 tokens (at least 512, at most 8, the last one split off
 * into its final 256 or so tokens when long enough), each range's
 * forward enters with the exact fp32 state the previous one left, and the
 * copies in, the forwards and the copies out run on three internal streams,
 * so the result is bitwise that of kda_chunk_fwd on the whole input.  With
 * segment ids it pipelines over two groups of heads (each group's copies
 * in, forward and copies out on an internal stream, the copies in chained
 * group after group), again bitwise equal to kda_chunk_fwd.  The work is
 * ordered after prior work on `stream`, and later work
 * on `stream` waits for it; the host outputs are valid once `stream`
 * synchronises.  `device_buffer` (caller-owned, 256-byte aligned,
 * zero-filled before its first use, reusable) holds the device copies and
 * the workspaces: kda_chunk_fwd_host_buffer_size bytes.  The
 * library creates its internal streams and events once per device and
 * keeps them for the process lifetime; enqueues are serialised by a mutex.
 * Errors: as kda_chunk_fwd (KDA_ERR_WORKSPACE for a small device_buffer,
 * KDA_ERR_ALIGNMENT for a misaligned one); a CUDA error while enqueuing
 * returns KDA_ERR_CUDA with part of the work possibly enqueued.
 */
KDA_API size_t kda_chunk_fwd_host_buffer_size(const kda_shape *s, int has_segment_ids);
KDA_API kda_status kda_chunk_fwd_host(const kda_shape *s, const void *q, const void *k,
                                      const void *v, const float *g, const float *beta,
                                      float scale, int chunk_size,
                                      const float *initial_state,
                                      const int32_t *segment_ids, void *o,
                                      float *final_state, void *device_buffer,
                                      size_t device_buffer_bytes, kda_stream_t stream);

/*
 * Backward of kda_chunk_fwd: the gradients of
 *     L = sum_t <d_o_t, o_t> + <d_final, final_state>
 * with respect to q, k, v, g, beta and initial_state, for the forward of page
 * "feat(kda): integrate KDA attention with tokamax backend and CP support",
 * section "Delta Rule formulation", with the packed runs of section "Public
 * API" (the pages' roadmap lists the backward as the next step; they print no
 * formula for it: this is reverse-mode differentiation of that recurrence).
 * Inputs as kda_chunk_fwd (q, k, v, g, beta, scale, chunk_size = 64,
 * initial_state or NULL = zeros, segment_ids or NULL), plus
 *   d_o        device [B,T,H,V] in s->qkv_dtype (the gradient of o);
 *   d_final    device float32 [B,H,K,V] or NULL (= zeros).
 * Outputs, all float32, caller-allocated:
 *   dq, dk, dg [B,T,H,K]; dv [B,T,H,V]; dbeta [B,T,H];
 *   d_initial  [B,H,K,V] or NULL (not wanted): the gradient with respect to
 *              the initial state (a zero one when initial_state is NULL).
 * Padding tokens get zero gradients; a row without a run passes d_final to
 * d_initial.  Supports K and V in {32, 64, 128}.
 * Two implementations; kda_chunk_bwd runs KDA_IMPL_AUTO (see _ex):
 *   tensor cores (KDA_IMPL_TC; KDA_IMPL_SPLIT names the same path): bf16
 *     q/k/v/d_o, K = V = 128, with or without segment_ids.  The chunked
 *     backward: the forward's per-chunk prep and its recurrence, which saves
 *     the state entering every chunk and U; the reverse chain of the state
 *     gradient (which saves dS' and dU per chunk); and a per-chunk kernel
 *     that forms every gradient of the chunk's tokens on tcgen05.
 *     Workspace: the chunk items and saves, 208.5 KiB per (chunk, head)
 *     plus 1 KiB (874 MB for B=1, T=8192, H=32).  With segment ids the
 *     workspace also holds the run list and chunk tables, and its items
 *     cover ceil(T/64) chunks per row plus one per run up to a bound:
 *     kda_chunk_bwd_workspace_size(_for) allows ceil(T/64) runs per row,
 *     kda_chunk_bwd_workspace_size_packed a bound of the caller's choice,
 *     and any workspace with room for ceil(T/64) chunks per row is accepted;
 *     when the runs of a call need more chunks than the workspace holds,
 *     the kernels compute nothing and set KDA_DEVICE_WORKSPACE in the status
 *     word (kda_read_device_status then returns KDA_ERR_WORKSPACE).
 *   CUDA cores (KDA_IMPL_SIMT): every supported shape, fp32.  It recomputes
 *     the states from checkpoints every 8 tokens and walks each (run, head,
 *     32-column value tile) backwards; its workspace holds the run list, the
 *     checkpoints and per-tile partial sums.
 * workspace: kda_chunk_bwd_workspace_size bytes (the AUTO choice), 256-byte
 * aligned, zero-filled before first use, reusable; its first word is the
 * device status word.  Errors as kda_chunk_fwd; the call is asynchronous
 * on `stream`.
 */
KDA_API size_t kda_chunk_bwd_workspace_size(const kda_shape *s, int has_segment_ids);
KDA_API kda_status kda_chunk_bwd(const kda_shape *s, const void *q, const void *k,
                                 const void *v, const float *g, const float *beta,
                                 float scale, int chunk_size, const float *initial_state,
                                 const int32_t *segment_ids, const void *d_o,
                                 const float *d_final, float *dq, float *dk, float *dv,
                                 float *dg, float *dbeta, float *d_initial, void *workspace,
                                 size_t workspace_bytes, kda_stream_t stream);

/*
 * Workspace bytes kda_chunk_bwd_ex needs for `impl`: KDA_IMPL_AUTO the
 * tensor-core size where that path applies, else the CUDA-core size;
 * KDA_IMPL_TC / KDA_IMPL_SPLIT 0 where the tensor-core path does not apply;
 * 0 for an invalid or unsupported shape.
 */
KDA_API size_t kda_chunk_bwd_workspace_size_for(const kda_shape *s, int has_segment_ids,
                                                kda_impl impl);
/*
 * Tensor-core backward workspace for inputs with segment ids and at most
 * max_runs_per_row runs in any row (0 for an invalid or unsupported shape
 * or max_runs_per_row < 1).
 */
KDA_API size_t kda_chunk_bwd_workspace_size_packed(const kda_shape *s, int max_runs_per_row);
/*
 * kda_chunk_bwd with an explicit implementation: KDA_IMPL_AUTO (tensor
 * cores where they apply, else CUDA cores), KDA_IMPL_SIMT, or KDA_IMPL_TC /
 * KDA_IMPL_SPLIT (KDA_ERR_UNSUPPORTED where the tensor-core path does not
 * apply); another value is KDA_ERR_INVALID_ARG.  The workspace must hold
 * kda_chunk_bwd_workspace_size_for(s, segment_ids != NULL, impl) bytes.
 */
KDA_API kda_status kda_chunk_bwd_ex(const kda_shape *s, const void *q, const void *k,
                                    const void *v, const float *g, const float *beta,
                                    float scale, int chunk_size, const float *initial_state,
                                    const int32_t *segment_ids, const void *d_o,
                                    const float *d_final, float *dq, float *dk, float *dv,
                                    float *dg, float *dbeta, float *d_initial,
                                    void *workspace, size_t workspace_bytes, kda_impl impl,
                                    kda_stream_t stream);

/*
 * A training step's forward and backward without repeating work: the
 * forward kda_chunk_fwd_save computes o and final_state exactly as
 * kda_chunk_fwd's split tensor-core path does (bit for bit) and also
 * leaves in `workspace` what the tensor-core backward reads (the per-chunk
 * items with T, A_kk and K e^G, and the state entering every chunk and U);
 * kda_chunk_bwd_from_saved then runs only the state-gradient chain and the
 * per-chunk gradient kernel on it, with results bit for bit those of
 * kda_chunk_bwd_ex(KDA_IMPL_TC) on the same inputs.
 * Supported: bf16 q/k/v/d_o, K = V = 128, with or without segment ids
 * (KDA_ERR_UNSUPPORTED otherwise).  Arguments as kda_chunk_fwd and
 * kda_chunk_bwd; the workspace (256-byte aligned, zero-filled before first
 * use) must hold kda_chunk_fwd_save_workspace_size bytes (the tensor-core
 * backward's size; with segment ids any workspace with room for ceil(T/64)
 * chunks per row is accepted and an overflow is reported as in
 * kda_chunk_bwd).  The caller passes kda_chunk_bwd_from_saved the same
 * shape, inputs (unchanged since the forward), segment ids and workspace
 * as the forward, with nothing written to the workspace in between; the
 * backward keeps the workspace's contents, so it may run again.  Both calls
 * are asynchronous on `stream`; errors as kda_chunk_fwd and kda_chunk_bwd.
 */
KDA_API size_t kda_chunk_fwd_save_workspace_size(const kda_shape *s, int has_segment_ids);
KDA_API kda_status kda_chunk_fwd_save(const kda_shape *s, const void *q, const void *k,
                                      const void *v, const float *g, const float *beta,
                                      float scale, int chunk_size,
                                      const float *initial_state,
                                      const int32_t *segment_ids, void *o,
                                      float *final_state, void *workspace,
                                      size_t workspace_bytes, kda_stream_t stream);
KDA_API kda_status kda_chunk_bwd_from_saved(const kda_shape *s, const void *q, const void *k,
                                            const void *v, const float *g, const float *beta,
                                            float scale, int chunk_size,
                                            const float *initial_state,
                                            const int32_t *segment_ids, const void *d_o,
                                            const float *d_final, float *dq, float *dk,
                                            float *dv, float *dg, float *dbeta,
                                            float *d_initial, void *workspace,
                                            size_t workspace_bytes, kda_stream_t stream);

/*
 * Test hook for failure detection (no counterpart in the pages): enqueues
 * one thread that waits, for at most `limit_cycles` SM clocks (1 .. about
 * 2^31), on an mbarrier nothing ever arrives at, using the bounded wait of
 * the tensor-core kernels; when the limit runs out it sets
 * KDA_DEVICE_TIMEOUT in the status word of `workspace` (a zero-filled
 * workspace of any size >= 256 bytes), which kda_read_device_status then
 * reports.  Nothing faults or hangs; the context stays usable.
 * KDA_ERR_INVALID_ARG for a NULL workspace or a limit out of range.
 */
KDA_API kda_status kda_selftest_wait_timeout(void *workspace, long long limit_cycles,
                                             kda_stream_t stream);

/* Static, NUL-terminated description of a status code. */
KDA_API const char *kda_status_string(kda_status status);

/* KDA_VERSION of the built library. */
KDA_API int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
