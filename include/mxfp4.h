/*
 * libmxfp4 -- MXFP4 linear layer on one NVIDIA GB300 (sm_103a).
 *
 * Computes C[M, N] = A[M, K] * B[N, K]^T with bf16 output, where A is a bf16
 * activation quantized on the fly to MXFP4 and B is a weight matrix quantized
 * to MXFP4 ahead of time.  MXFP4 (OCP Microscaling v1.0): each run of 32
 * consecutive K elements of a row shares one E8M0 scale byte (value
 * 2^(byte - 127)); each element is an E2M1 code (sign | 2-bit exponent |
 * 1-bit mantissa; magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6), two codes per byte,
 * the even K index in the low nibble.  This is the problem of the
 * amd-mxfp4-mm leaderboard (kernelindex.com submissions 748756, 721672,
 * 754569, 755056, 733989): `custom_kernel((A, B, B_q, B_shuffle,
 * B_scale_sh)) -> C`.
 *
 * Conventions for every call:
 *   - Pointers marked "device" are CUDA device pointers on the current device;
 *     the caller allocates and owns every buffer.  No call allocates device
 *     memory, so every compute call may be captured in a CUDA graph.
 *   - Compute calls are asynchronous on `stream` (NULL = legacy default stream)
 *     and return after the launch; their results are ready when the stream is.
 *   - Arguments are checked on the host before anything is launched; a call
 *     that returns an error status has launched nothing.  There is no fallback
 *     path: a shape or alignment outside the contract is an error.
 *   - Sizes are int64_t element counts.  K must be a positive multiple of 32.
 *     Every device pointer must be 16-byte aligned.
 *   - Device-side waits are bounded (about one second by default).  A wait
 *     that runs out sets the library's device error word and the kernel
 *     finishes without its result; read the word with mxfp4_device_error().
 *   - The library keeps device arrays of its own (the error word, and the
 *     scratch of mxfp4_quant_gemm_static_scratch) and resolves their device
 *     addresses once per device.  A cudaDeviceReset() in the process
 *     invalidates those addresses: do not call the library after one.
 */
#ifndef MXFP4_H_
#define MXFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream). */
typedef struct CUstream_st* mxfp4_stream_t;

typedef enum {
  MXFP4_OK = 0,
  MXFP4_ERR_INVALID_ARG = 1,        /* null pointer, non-positive size, K % 32 != 0, bad plan */
  MXFP4_ERR_UNSUPPORTED_SHAPE = 2,  /* a size beyond the library's limits */
  MXFP4_ERR_MISALIGNED = 3,         /* a pointer or leading dimension not 16-byte aligned */
  MXFP4_ERR_WORKSPACE_TOO_SMALL = 4,/* a workspace smaller than the chosen route needs */
  MXFP4_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed */
  MXFP4_ERR_DEVICE_TIMEOUT = 6,     /* a device-side bounded wait ran out */
  MXFP4_ERR_UNSUPPORTED_DEVICE = 7  /* the current device is not sm_103 */
} mxfp4_status_t;

/* Tile plan of one GEMM launch (see mxfp4_gemm_plan). */
typedef struct {
  int32_t block_m;    /* activation rows per CTA = the MMA's N: 16, 32, 64, 128 or 256 */
  int32_t splits;     /* K splits per output tile = CTAs per thread-block cluster, 1..8 */
  int32_t stages;     /* shared-memory pipeline depth in K tiles of 256 */
  int32_t k_tiles_per_split;
  int32_t grid_x, grid_y, grid_z; /* splits, N tiles of 128, M tiles of block_m */
  int32_t threads;    /* threads per CTA */
  int32_t smem_bytes; /* dynamic shared memory per CTA */
  int32_t tmem_cols;  /* tensor-memory columns allocated per CTA */
  int32_t two_pass;   /* mxfp4_gemm_plan, fused entry: 1 if, given mxfp4_workspace_bytes() of
                         workspace, it quantizes A into the workspace and runs the GEMM on
                         codes (this plan then describes that GEMM) */
  int32_t accumulators; /* independent fp32 accumulator tiles in tensor memory: 1, 2 or 4
                           (K step g goes to tile g mod accumulators; summed in the epilogue) */
  int32_t share;      /* fused entry: CTAs of neighbouring N tiles that quantize the activation once
                         between them (each a share of the K tiles, pushed into the others' shared
                         memory); 1 = each CTA quantizes its own, 0 = the default choice.  The
                         cluster is splits x share CTAs */
} mxfp4_plan_t;

/* ---------------------------------------------------------------------------
 * mxfp4_quantize -- A (bf16) -> MXFP4 codes + E8M0 scales.
 *
 * The rule of `hw_pack_mxfp4` (submission 748756) and "Software MXFP4 quant"
 * (submission 755056): per row and 32-element block, amax = max |x|;
 * u = (bits(amax) + 0x200000) & 0xFF800000; s = clamp(exponent(u) - 129,
 * -127, 127); scale byte = s + 127; each element x -> E2M1(x * 2^-s) with
 * round-to-nearest-even, saturating at 6, sign kept (so -0 -> 0x8).
 *
 *   A   device, bf16 [M, lda] row-major (first K columns used); lda % 8 == 0
 *   Aq  device, uint8 [M, K/2] row-major, byte = code[2i] | code[2i+1] << 4
 *   As  device, uint8 [M, K/32] row-major
 * M >= 1.  Returns MXFP4_OK or an error status (nothing launched).
 * ------------------------------------------------------------------------- */
mxfp4_status_t mxfp4_quantize(const void* A, int64_t M, int64_t K, int64_t lda, void* Aq, void* As,
                              mxfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * Packed weights: the one-time relayout of a pre-quantized B (the pages cache
 * such a relayout per weight, e.g. the linearised-weight cache of submission
 * 748756) into the layout the GEMM streams with TMA:
 *   - codes: [roundup(N,128), K/2] bytes, rows >= N zero;
 *   - scales: for each 128-row N tile and 256-wide K tile, 1024 bytes: two
 *     512-byte chunks (K sub-blocks of 128), byte (r%32)*16 + (r/32)*4 + j for
 *     tile row r and scale j = 0..3 of the chunk; padding scales are 0.
 * The buffer is opaque to callers; its size is mxfp4_packed_weight_bytes().
 * ------------------------------------------------------------------------- */
size_t mxfp4_packed_weight_bytes(int64_t N, int64_t K);

/*   Bq      device, uint8 [N, K/2] (natural layout, as mxfp4_quantize writes it)
 *   Bs      device, uint8 [N, K/32]
 *   Bpacked device, mxfp4_packed_weight_bytes(N, K) bytes, written entirely. */
mxfp4_status_t mxfp4_pack_weights(const void* Bq, const void* Bs, int64_t N, int64_t K, void* Bpacked,
                                  mxfp4_stream_t stream);

/* The same packed buffer from the weight layouts the pages' harness hands out
 * (`custom_kernel((A, B, B_q, B_shuffle, B_scale_sh))`), so that tuple runs as
 * it is:
 *   B_shuffle   device, uint8 [N, K/2] bytes in the preshuffled layout of
 *               `materialize_linear_weight_layout` (submission 748756):
 *               16-row x 16-byte subtiles; natural byte (n, kb) at
 *               ((n/16 * Kh/32 + kb/32) * 2 + (kb%32)/16) * 256 + (n%16) * 16 + kb%16,
 *               Kh = K/2.
 *   B_scale_sh  device, uint8, the e8m0 shuffle (`materialize_linear_scale_layout`;
 *               the shuffled-scale store of submission 755056): scale (n, g) at
 *               (n/32) * 32 * Gp + (g/8) * 256 + (g%4) * 64 + (n%16) * 4
 *               + ((g%8)/4) * 2 + (n%32)/16, Gp = K/32 rounded up to 8; at least
 *               roundup(N, 32) * Gp bytes (aiter pads the rows to 256).
 * N % 16 == 0 and K % 64 == 0 (the layouts' own granularity). */
mxfp4_status_t mxfp4_pack_weights_shuffled(const void* B_shuffle, const void* B_scale_sh, int64_t N, int64_t K,
                                           void* Bpacked, mxfp4_stream_t stream);

/* Inverse of mxfp4_pack_weights (for checking a packed buffer). */
mxfp4_status_t mxfp4_unpack_weights(const void* Bpacked, int64_t N, int64_t K, void* Bq, void* Bs,
                                    mxfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * GEMM.  C[m, n] = sum_k deq(A)[m, k] * deq(B)[n, k], block-scaled FP4 x FP4
 * products accumulated in fp32 (the pages' `tl.dot_scaled(a, a_scale, "e2m1",
 * b, b_scale, "e2m1", acc)`), K splits summed in fp32 in a fixed order
 * (deterministic), rounded to bf16 (nearest even).
 *
 *   Aq, As   device, the outputs of mxfp4_quantize for A [M, K]
 *   A        device, bf16 [M, lda]; lda % 8 == 0 (fused entry only)
 *   Bpacked  device, the output of mxfp4_pack_weights for the same N, K
 *   C        device, bf16 [M, N] row-major, fully overwritten
 *   ws, ws_bytes  device scratch, optional (NULL, 0 is always valid).
 *            mxfp4_gemm needs none: it accepts and ignores any ws, ws_bytes.
 *            mxfp4_quant_gemm chooses its route by them:
 *              - ws_bytes == 0: the single fused kernel, for every M;
 *              - ws_bytes > 0 and mxfp4_workspace_bytes(M, N, K) non-zero
 *                (M >= 64, except where M <= 128 and 2*M*K*ceil(N/128)
 *                <= 5 MiB, and the shapes whose tuned plan is the single
 *                kernel): the two-pass route -- A quantized into the
 *                workspace by mxfp4_quantize, then the GEMM on the codes, two
 *                launches that overlap; faster than the single kernel once M
 *                is large, because that kernel re-reads the bf16 activation
 *                in every 128-row weight tile.  ws_bytes below
 *                mxfp4_workspace_bytes(M, N, K) returns
 *                MXFP4_ERR_WORKSPACE_TOO_SMALL, a ws that is not 16-byte
 *                aligned MXFP4_ERR_MISALIGNED (nothing launched);
 *              - ws_bytes > 0 otherwise: the single fused kernel (ws unused);
 *              - ws == NULL with ws_bytes > 0: MXFP4_ERR_INVALID_ARG.
 *            The workspace is overwritten; calls that share one must be
 *            ordered.
 * M, N >= 1.  Returns MXFP4_OK or an error status (nothing launched).
 * ------------------------------------------------------------------------- */
/* Workspace that lets mxfp4_quant_gemm take its two-pass route (0 when the
 * single fused kernel is best, or for invalid sizes): M*K/2 + M*K/32 bytes,
 * each part rounded up to 256. */
size_t mxfp4_workspace_bytes(int64_t M, int64_t N, int64_t K);

mxfp4_status_t mxfp4_gemm(const void* Aq, const void* As, const void* Bpacked, void* C, int64_t M,
                          int64_t N, int64_t K, void* ws, size_t ws_bytes, mxfp4_stream_t stream);

/* The fused entry: quantizes A inside the GEMM kernel (no global Aq/As), with
 * the same rule and bit-identical codes as mxfp4_quantize (or, given a
 * workspace for M >= 64, in a separate pass; see ws above). */
mxfp4_status_t mxfp4_quant_gemm(const void* A, int64_t lda, const void* Bpacked, void* C, int64_t M,
                                int64_t N, int64_t K, void* ws, size_t ws_bytes,
                                mxfp4_stream_t stream);

/* The fused entry for activations and results in host memory: uploads A
 * (host bf16 [M, lda_host]) into A_dev (device bf16 [M, lda_dev]), runs
 * mxfp4_quant_gemm on it (C_dev, ws as there) and delivers the result to both
 * C_dev and C_host (host bf16 [M, N]) -- asynchronous operations on `stream`,
 * issued by one call.  The caller owns every buffer; host buffers should be
 * pinned (page-locked) for the transfers to be asynchronous.
 *   - A_host pinned and addressable by the device (mapped host memory) with
 *     16-byte aligned rows (lda_host a multiple of 8): uploaded by the
 *     library's copy kernel, SM threads reading host memory over the host
 *     link; otherwise by cudaMemcpy2DAsync.
 *   - C_host mapped and 16-byte aligned: written by the GEMM kernel itself,
 *     beside C_dev (no download pass); otherwise C_dev is downloaded by
 *     cudaMemcpyAsync after the GEMM.
 * The upload reads A_host as soon as its kernel starts (under programmatic
 * launch possibly while the previous kernel on the stream still runs), so
 * A_host must hold the input when the call is made -- the same rule as for
 * any asynchronous copy from it.  C_host is complete when the stream is.  All
 * checks precede the upload: an error launches nothing. */
mxfp4_status_t mxfp4_quant_gemm_host(const void* A_host, int64_t lda_host, void* A_dev, int64_t lda_dev,
                                     const void* Bpacked, void* C_dev, void* C_host, int64_t M, int64_t N,
                                     int64_t K, void* ws, size_t ws_bytes, mxfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * mxfp4_quant_gemm_static_scratch -- the fused layer without any allocation.
 *
 * The pages have no counterpart: this exists for callers that cannot allocate
 * device memory -- a plugin inside a host framework that reserves all device
 * memory up front and forbids allocation afterwards, or code that must not
 * call cudaMalloc because it synchronises the device -- and so cannot give
 * mxfp4_quant_gemm the workspace of its two-pass route.  This call always runs
 * that route (mxfp4_quantize into scratch, then mxfp4_gemm on the codes) with
 * the scratch in a 4 MiB device array the library owns: every GPU that loads
 * the library holds it until the process exits.  The caller passes only the
 * inputs and the output, as for mxfp4_quant_gemm (A bf16 [M, lda], Bpacked, C
 * bf16 [M, N]); nothing is allocated.
 *   - Sizes whose codes and scales (M*K/2 + M*K/32 bytes, each rounded up to
 *     256) exceed 4 MiB return MXFP4_ERR_UNSUPPORTED_SHAPE, launching nothing;
 *     mxfp4_last_error_string() then names the limit.
 *   - The first call on a device resolves the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Every call shares the one array, which keeps the last call's contents
 *     (nothing in it needs clearing: each call overwrites what it reads).
 *     Calls that can overlap on the GPU -- on streams not ordered with each
 *     other -- race on it.
 * For M < 64, mxfp4_quant_gemm with no workspace needs no scratch at all and
 * is faster. */
mxfp4_status_t mxfp4_quant_gemm_static_scratch(const void* A, int64_t lda, const void* Bpacked, void* C,
                                               int64_t M, int64_t N, int64_t K, mxfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * mxfp4_quant_gemm_chain -- several dependent layers in one launch.
 *
 * Layer l computes C_l = quant(X_l) * B_l^T (the fused layer above), with
 * X_0 = A and X_l = C_{l-1} for l >= 1: K_0 = K, K_l = N_{l-1}.  The pages run
 * one quantize + GEMM per layer and find most of each call's time in the
 * per-launch cost (submission 733989, "PROFILING"; submission 755056 captures
 * its launches in a CUDA graph for the same reason); here one persistent
 * kernel runs every layer: its CTAs stay resident, each layer waits only for
 * the K tiles of its input that it reads (bounded device-side waits on
 * completion counters), the next layer's weights load while the current
 * layer finishes, and each layer's epilogue quantizes its own bf16 output
 * for the next layer (bit-identical to mxfp4_quantize of C_l).  The first
 * layer's activation is quantized once, shared by all CTAs.
 *
 *   A        device, bf16 [M, lda]; lda >= K, lda % 8 == 0
 *   M, K     rows of every X_l / C_l, and the first layer's K (K % 32 == 0)
 *   num_layers  1 .. 16
 *   Bpacked  host array of num_layers device pointers: the packed weights
 *            [N_l, K_l] (mxfp4_pack_weights)
 *   N        host array of num_layers output widths; N_l % 32 == 0 for every
 *            layer but the last (N_l is the next layer's K)
 *   C        host array of num_layers device pointers, bf16 [M, N_l]
 *            row-major, every layer's output written
 *   ws, ws_bytes  device workspace of at least
 *            mxfp4_chain_workspace_bytes(M, K, num_layers, N) bytes, 256-byte
 *            aligned, and ZERO-INITIALISED before its first use (cudaMemset).
 *            It holds each layer's activation codes, split-K partials and
 *            the completion counters; every call returns the counters to
 *            zero, so one zeroing serves any number of calls with the same
 *            workspace.  Calls sharing a workspace must be ordered (one
 *            stream).  If a call's device-side wait runs out (see
 *            mxfp4_device_error), zero the workspace again.  A workspace that
 *            was not zeroed makes the kernel's waits run out and report,
 *            instead of producing a wrong result.
 * Rows of C_l are identical in meaning to mxfp4_quant_gemm's on the same
 * input; values agree within fp32 summation order (K splits may differ).
 * Every CTA must be resident at once (the grid is at most one wave of the
 * device); kernels of other streams that hold SMs for longer than the wait
 * limit make the call report a timeout.  Errors as for the other entries:
 * nothing launched unless MXFP4_OK. */
size_t mxfp4_chain_workspace_bytes(int64_t M, int64_t K, int32_t num_layers, const int64_t* N);

mxfp4_status_t mxfp4_quant_gemm_chain(const void* A, int64_t lda, int64_t M, int64_t K, int32_t num_layers,
                                      const void* const* Bpacked, const int64_t* N, void* const* C, void* ws,
                                      size_t ws_bytes, mxfp4_stream_t stream);

/* The plan of a multi-layer launch: per layer its K split count (splits, a
 * host array of num_layers, may be NULL), the grid size and the rows of
 * activation per CTA.  Host only, launches nothing. */
mxfp4_status_t mxfp4_chain_plan(int64_t M, int64_t K, int32_t num_layers, const int64_t* N, int32_t* splits,
                                int32_t* grid, int32_t* block_m);

/* The plan the two GEMM entries would use for (M, N, K); fused != 0 for the
 * fused entry.  Host only, launches nothing. */
mxfp4_status_t mxfp4_gemm_plan(int64_t M, int64_t N, int64_t K, int fused, mxfp4_plan_t* plan);

/* The GEMM entries with an explicit plan: only block_m, splits, stages,
 * accumulators and share (0 = the default choice) are read (the rest is
 * derived; a plan with share > 1 takes a stage per K tile); a plan
 * the device cannot run is rejected with
 * MXFP4_ERR_INVALID_ARG.  fused != 0 reads A/lda, else Aq/As. */
mxfp4_status_t mxfp4_gemm_with_plan(const void* A_or_Aq, int64_t lda, const void* As,
                                    const void* Bpacked, void* C, int64_t M, int64_t N, int64_t K,
                                    int fused, const mxfp4_plan_t* plan, mxfp4_stream_t stream);

/* ---------------------------------------------------------------------------
 * Errors and diagnostics.
 * ------------------------------------------------------------------------- */
const char* mxfp4_status_string(mxfp4_status_t status);

/* A message for the last MXFP4_ERR_CUDA status returned on the calling
 * thread (the CUDA call and its error), or for the last
 * MXFP4_ERR_UNSUPPORTED_SHAPE that mxfp4_quant_gemm_static_scratch returned
 * because its size limit was exceeded; "" if none.  Valid until the thread's
 * next call that sets it. */
const char* mxfp4_last_error_string(void);

/* Synchronises `stream`, then reads the device error word (0 = no device-side
 * failure since the last reset) into *code and, if reset != 0, clears it.
 * Returns MXFP4_ERR_DEVICE_TIMEOUT if the word is non-zero, else MXFP4_OK. */
mxfp4_status_t mxfp4_device_error(mxfp4_stream_t stream, int reset, uint32_t* code);

/* Limit, in nanoseconds, of every device-side wait in kernels launched after
 * this call (default 1e9; 0 restores the default). */
mxfp4_status_t mxfp4_set_wait_timeout_ns(uint64_t ns);

/* How a GEMM call may overlap the kernel before it on the same stream
 * (programmatic dependent launch):
 *   0  no overlap: the GEMM starts after the previous kernel has finished;
 *   1  the GEMM may start early, but until the previous kernel has completed
 *      it only sets up and prefetches its weight and activation bytes into L2
 *      (L2 is coherent, so this never reads stale data);
 *   2  as 1, and the weight codes and scales are also loaded into shared
 *      memory before the previous kernel has completed.  Contract: the packed
 *      weight buffer is not written by the kernel that immediately precedes
 *      the GEMM on its stream (weights are read-only parameters; none of this
 *      library's kernels writes a weight buffer it is not given as an output,
 *      and a kernel that does not use programmatic launch has always
 *      completed before the GEMM starts).  A GEMM lets the next kernel start
 *      as soon as it has itself started, so a chain of calls can run several
 *      grids ahead;
 *   3  (default) as 2, but a GEMM lets the next kernel start only once its
 *      own wait for the previous kernel has ended and its activation loads
 *      are under way: at most one grid runs ahead, and the grids waiting
 *      early no longer crowd the running one's SMs (measured faster on GB300
 *      for every shape with few K tiles).
 * mxfp4_quantize follows modes 1 and 2 likewise: it may start early, but reads
 * A and writes its outputs only after the previous kernel has completed.
 * In every mode the activation is read, and C written, only after the
 * previous kernel has completed.  Back-to-back calls then overlap one call's
 * set-up and weight streaming with the previous call's tail. */
mxfp4_status_t mxfp4_set_programmatic_launch(int mode);

/* Diagnostic: launches one tiny kernel whose wait can never complete (an
 * mbarrier nothing arrives on) and that therefore gives up after the current
 * wait limit and sets the device error word.  Lets a caller check that bounded
 * waits end and report instead of hanging. */
mxfp4_status_t mxfp4_diag_wait_timeout(mxfp4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_H_ */
