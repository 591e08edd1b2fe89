/*
 * fa.h — C ABI of the GB300 (sm_103a) attention forward library, libfa.so.
 *
 * The operation is exact scaled-dot-product attention,
 *     O = softmax(scale * Q K^T [+ causal mask]) V,
 * the problem statement of the concept card "FlashAttention 2 + 3 —
 * speicherbewusste Attention-Kernels" (section "Kernpunkte": the same output as
 * softmax(QK^T/sqrt(d)) V, with the N x N matrix never written to HBM) and of the
 * "Flash Attention" glossary (section "/01 Was ist Flash Attention?"), computed
 * tile by tile with an online softmax (concept card, "Begriffe auf dieser Seite",
 * Online-Softmax).  Each call also writes the per-row log-sum-exp.  The FP8 entry
 * points follow the FlashAttention-3 news piece ("Drei technische Hebel", item 3:
 * block-wise 8-bit quantisation with a Hadamard transform) and the concept card's
 * absmax scaling ("Kernpunkte", FP8 item).
 *
 * Conventions shared by every entry point
 *   - Tensors are contiguous, row-major [B, H, N, d] with d innermost; LSE is
 *     [B, H, N] float32; block scales are [B, H, ceil(N/64)] float32.
 *   - Data pointers are DEVICE pointers owned by the caller, 16-byte aligned
 *     (LSE and scales 4-byte aligned).  The library keeps no pointer after the
 *     call returns and allocates no per-call memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls are asynchronous on that stream; nothing synchronises
 *     except fa_last_device_status.
 *   - The current CUDA device must be an sm_103 GPU.
 *   - Errors are returned as fa_status codes, never thrown.  Argument errors are
 *     detected on the host before any device work is enqueued.
 *   - Causal masking is top-left aligned: query row i sees keys 0..i.
 *   - Supported: B, H, N >= 1; d in {64, 128}; B*H*N*d < 2^40.
 *   - Every pipeline wait inside a kernel is bounded (2 s by default, the
 *     environment variable FA_TIMEOUT_MS overrides it).  A kernel whose wait gives
 *     up sets a bit in the device status word and leaves early: its outputs are
 *     then UNDEFINED, yet the call that launched it has already returned FA_OK.
 *     Callers that must know call fa_last_device_status after the work they care
 *     about (it synchronises and returns FA_ERR_DEVICE_TIMEOUT if any wait gave up).
 *   - Per-device state (the status word's address, fa_decode_noalloc's scratch
 *     address, fa_fwd_host's copy streams) is looked up once per device in the
 *     context current at the first call, normally the device's primary context.
 *     Do not call the library after cudaDeviceReset, or from another context on
 *     a device it has already been used on.
 */
#ifndef FA_GB300_H_
#define FA_GB300_H_

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FA_F16 = 0, FA_BF16 = 1 } fa_dtype;

typedef enum {
  FA_OK = 0,
  FA_ERR_NULL = -1,            /* a required pointer is NULL */
  FA_ERR_ALIGN = -2,           /* a pointer is not aligned as stated above */
  FA_ERR_SHAPE = -3,           /* B, H or N out of range, or sizes overflow */
  FA_ERR_UNSUPPORTED = -4,     /* head dim, dtype or flag value not supported */
  FA_ERR_LAUNCH = -5,          /* the kernel launch was rejected by the runtime */
  FA_ERR_DEVICE_TIMEOUT = -6,  /* a kernel gave up on a pipeline wait (see fa_last_device_status) */
  FA_ERR_ARCH = -7,            /* the current device is not an sm_103 GPU */
  FA_ERR_CUDA = -8,            /* another CUDA runtime or driver call failed */
  FA_ERR_WORKSPACE = -9        /* workspace missing or smaller than fa_decode_workspace_size */
} fa_status;

/*
 * Attention forward in f16 or bf16.
 *   q, k, v : [B, H, N, d] of `dtype` (FA_F16 or FA_BF16)
 *   o       : [B, H, N, d] of `dtype`, written
 *   lse     : [B, H, N] float32, written: natural log of sum_j exp(scale * q_i.k_j)
 *             over the visible keys; may be NULL (not written)
 *   scale   : multiplies Q K^T (1/sqrt(d) gives the textbook definition); finite and > 0
 *   causal  : 0 or 1
 * Accumulation is fp32; the softmax weights are rounded to `dtype` before the
 * weighted sum over V, and O is rounded to `dtype` once at the end.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, int dtype, void* stream);

/*
 * fa_fwd computed by pairs of CTAs on two SMs (a cluster of two), with M = 256 tensor-core
 * tiles issued for both SMs by one thread (tcgen05 cta_group::2): each SM holds half of
 * every K and V tile, so a key tile costs each SM half the shared memory.  This is the
 * larger tile the FlashAttention-3 news piece's levers point at ("Drei technische
 * Hebel", items 1-2); the operation and the results' accuracy are fa_fwd's.
 * Arguments, layout, ownership and errors as fa_fwd; supported: d == 128 only (other
 * head dims return FA_ERR_UNSUPPORTED).
 */
int fa_fwd_2cta(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                int d, float scale, int causal, int dtype, void* stream);

/*
 * fa_fwd on HOST buffers, end to end: copies Q, K, V to the device, computes, and copies
 * O (and LSE) back, with the copies of one chunk of heads overlapped with the
 * computation of the next (a runtime convenience; the pages' operation is fa_fwd's).
 *   q, k, v, o : [B, H, N, d] of `dtype` in host memory (pinned memory lets the copies
 *                run asynchronously; pageable memory works, without overlap)
 *   lse        : [B, H, N] float32 in host memory, or NULL
 *   chunks     : number of equal head chunks (at most 32 and B*H); 0 picks chunks of
 *                1, 2, 4, ... heads up to B*H/8 and back down to 1 at the end, so that
 *                little crosses the link while nothing computes
 *   workspace  : DEVICE scratch of at least fa_fwd_host_workspace_size() bytes,
 *                256-byte aligned, owned by the caller; calls sharing one workspace must
 *                be on one stream (the copies wait for earlier work on `stream`)
 * Asynchronous: the results are on the host once `stream` reaches this point
 * (synchronise it).  Two copy streams, two compute streams (consecutive chunks run on
 * them in turn, so that one chunk's grid fills the SMs the previous one's last CTAs
 * leave idle) and a few events per device are created on the first call there;
 * concurrent calls from several host threads are serialised while they enqueue.
 * Errors as fa_fwd, plus FA_ERR_WORKSPACE.
 */
int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                float scale, int causal, int dtype, int chunks, void* workspace,
                unsigned long long workspace_bytes, void* stream);

/* Device scratch fa_fwd_host needs: Q, K, V, O and LSE on the device, 256-byte aligned each. */
int fa_fwd_host_workspace_size(int B, int H, int N, int d, unsigned long long* bytes);

/*
 * FP8 prologue: optional Hadamard rotation along d, block absmax, E4M3 quantisation.
 *   x        : [B, H, N, d] bfloat16 input
 *   x8       : E4M3 output, [B, H, N, d]; with transpose_out = 1 it is [B, H, d, N]
 *              instead (the layout fa_fwd_fp8 wants for V), which needs N % 16 == 0
 *   scale    : [B, H, ceil(N/64)] float32, written: s = absmax/448 of the (rotated)
 *              64-row block, 1 for an all-zero block; x8 = e4m3_rn_satfinite(x/s)
 *   hadamard : 1 applies x -> x H_d / sqrt(d) (Sylvester order) before the absmax;
 *              0 does not.  Use 1 for Q and K only, never for V.
 * Errors: FA_ERR_NULL, FA_ERR_SHAPE, FA_ERR_UNSUPPORTED, FA_ERR_ALIGN (x, x8 16-byte
 * aligned, scale 4-byte), FA_ERR_ARCH, FA_ERR_LAUNCH.  The kernel's waits for its
 * bulk copies are bounded; one that gives up ORs 1 into the device status word (and
 * 8 if a copy had still not landed when its CTA left); see fa_last_device_status.
 */
int fa_quantize_fp8(const void* x, void* x8, float* scale, int B, int H, int N, int d, int hadamard,
                    int transpose_out, void* stream);

/*
 * fa_quantize_fp8 with two variants of the prologue (steps beyond the pages, which
 * name only a "Hadamard-Transformation" and "Absmax" scaling):
 *   sign_flips_lo/hi : randomised rotation x -> (x * sigma) H_d / sqrt(d), where bit c
 *                      of the 128-bit mask (lo = bits 0..63, hi = bits 64..127) sets
 *                      sigma_c = -1.  Use the same mask for Q and K: scores are
 *                      unchanged, so fa_fwd_fp8 needs nothing else.  Must be 0 when
 *                      hadamard = 0, and hi must be 0 for d = 64 (FA_ERR_UNSUPPORTED).
 *   per_head         : 1 takes one absmax over all N rows of each (b, h) and writes it
 *                      to every block entry of `scale` (the layout fa_fwd_fp8 reads);
 *                      0 is the per-64-row-block scale of fa_quantize_fp8.  Per-head
 *                      reads x twice (absmax pass, then quantisation pass).
 * Other arguments and errors as fa_quantize_fp8.
 */
int fa_quantize_fp8_ex(const void* x, void* x8, float* scale, int B, int H, int N, int d, int hadamard,
                       unsigned long long sign_flips_lo, unsigned long long sign_flips_hi, int per_head,
                       int transpose_out, void* stream);

/*
 * The whole FP8 prologue in one launch: Q and K quantised as fa_quantize_fp8 with
 * `hadamard`, V quantised without rotation and written transposed (transpose_out = 1).
 * The three tensors' blocks form one sequence of work for one persistent grid, so the
 * launch has one ramp and one tail instead of three.  Codes and scales are bitwise those
 * of the three separate calls.
 *   q, k, v          : [B, H, N, d] bfloat16
 *   q8, k8           : [B, H, N, d] E4M3;  v8t : [B, H, d, N] E4M3
 *   q_scale, k_scale, v_scale : [B, H, ceil(N/64)] float32, written
 * Needs N % 16 == 0.  Errors as fa_quantize_fp8.
 */
int fa_quantize_fp8_qkv(const void* q, const void* k, const void* v, void* q8, void* k8, void* v8t,
                        float* q_scale, float* k_scale, float* v_scale, int B, int H, int N, int d,
                        int hadamard, void* stream);

/*
 * Attention forward from E4M3 inputs produced by fa_quantize_fp8.
 *   q8, k8   : [B, H, N, d] E4M3 (rotated by the same Hadamard matrix, or both not)
 *   v8t      : [B, H, d, N] E4M3 (V quantised with transpose_out = 1, not rotated)
 *   q_scale, k_scale, v_scale : [B, H, ceil(N/64)] float32 block scales
 *   o        : [B, H, N, d] bfloat16, written;  lse as for fa_fwd (may be NULL)
 *   hadamard : records whether Q and K were rotated (0 or 1); (QH)(KH)^T = QK^T,
 *              so it changes no arithmetic here and is only validated
 * Supported: d == 128, N % 16 == 0, non-causal or causal.
 */
int fa_fwd_fp8(const void* q8, const void* k8, const void* v8t, void* o, float* lse, int B, int H,
               int N, int d, float scale, int causal, const float* q_scale, const float* k_scale,
               const float* v_scale, int hadamard, void* stream);

/*
 * The FP8 mode end to end on HOST buffers: bf16 Q, K, V in, bf16 O (and LSE) out.  On the
 * device, each chunk of heads runs the whole FP8 path of the news piece ("Drei
 * technische Hebel", item 3): fa_quantize_fp8_qkv (Q and K rotated when `hadamard` is 1,
 * V transposed, never rotated), then fa_fwd_fp8.  The copies of one chunk overlap
 * the computation of the next, as in fa_fwd_host (a runtime convenience).
 *   q, k, v, o : [B, H, N, d] bfloat16 in host memory (pinned lets the copies overlap)
 *   lse        : [B, H, N] float32 in host memory, or NULL
 *   hadamard   : 0 or 1
 *   chunks     : number of equal head chunks (at most 32 and B*H); 0 picks chunks of
 *                1, 2, 4, ... heads up to B*H/8 and back down to 1 at the end, so that
 *                little crosses the link while nothing computes
 *   workspace  : DEVICE scratch of at least fa_fwd_fp8_host_workspace_size() bytes,
 *                256-byte aligned, owned by the caller; calls sharing one workspace must
 *                be on one stream
 * Supported: d == 128, N % 16 == 0.  Asynchronous like fa_fwd_host; errors as
 * fa_fwd_fp8 and fa_quantize_fp8, plus FA_ERR_WORKSPACE.
 */
int fa_fwd_fp8_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                    int d, float scale, int causal, int hadamard, int chunks, void* workspace,
                    unsigned long long workspace_bytes, void* stream);

/* Device scratch fa_fwd_fp8_host needs: the bf16 inputs and output, the E4M3 codes, the
 * block scales and the LSE, 256-byte aligned each. */
int fa_fwd_fp8_host_workspace_size(int B, int H, int N, int d, unsigned long long* bytes);

/*
 * Attention of a few query rows against a long key cache (one decode step): the
 * same definition as fa_fwd, for the last N_q positions of a sequence of N_k keys
 * (the concept card's problem statement, "Kernpunkte", applied to the KV cache of
 * "Begriffe auf dieser Seite").  With causal = 1, query row i sees keys
 * 0 .. N_k - N_q + i (bottom-right alignment); with 0, all keys.
 *   q          : [B, H, N_q, d] of `dtype`, 1 <= N_q <= 16, N_q <= N_k
 *   k, v       : [B, H, N_k, d] of `dtype`
 *   o, lse     : [B, H, N_q, d] of `dtype` and [B, H, N_q] float32 (lse may be NULL)
 *   num_splits : key chunks per head processed in parallel and merged by log-sum-exp;
 *                0 picks the count that best fills whole waves of CTAs on this GPU
 *                (chunks of at least 256 keys, at most 4 MiB of scratch)
 *   workspace  : device scratch of at least fa_decode_workspace_size() bytes, 256-byte
 *                aligned, owned by the caller; may be NULL when that size is 0.  Its
 *                contents on entry do not matter; calls sharing one workspace must not
 *                overlap on the GPU.
 * Computed on the CUDA cores (the work is a stream over K and V, HBM-bound).
 */
int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
              int Nk, int d, float scale, int causal, int dtype, int num_splits, void* workspace,
              unsigned long long workspace_bytes, void* stream);

/* Scratch bytes fa_decode needs for these sizes on the current device (0 if none). */
int fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits,
                             unsigned long long* bytes);

/*
 * Backward pass: dQ, dK, dV of fa_fwd's output for an upstream gradient dO.  The
 * pages name the backward pass as where FlashAttention-2 parallelises better (the
 * concept card "FlashAttention 2 + 3 — speicherbewusste Attention-Kernels", section
 * "Kernpunkte") but print no formula: the gradient is the calculus of fa_fwd's
 * definition, with P recomputed tile by tile from the saved LSE,
 *   P = exp(scale * Q K^T - LSE),  D_i = sum_c dO_ic O_ic,  dS = P * (dO V^T - D),
 *   dV = P^T dO,  dQ = scale * dS K,  dK = scale * dS^T Q.
 *   q, k, v, o, dout : [B, H, N, d] of `dtype`; o and lse are fa_fwd's outputs for
 *                      the same q, k, v, scale and causal (lse must not be NULL there)
 *   dq, dk, dv       : [B, H, N, d] of `dtype`, written
 *   workspace        : device scratch of at least fa_bwd_workspace_size() bytes,
 *                      256-byte aligned, owned by the caller; contents on entry do not
 *                      matter; calls sharing one workspace must not overlap on the GPU
 * Same support as fa_fwd (d in {64, 128}, f16/bf16, causal 0 or 1, any N >= 1).  P
 * and dS are rounded to `dtype` before their MMAs and the results once at the end;
 * accumulation is fp32.  No atomics: results are bitwise reproducible.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
           void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, int dtype,
           void* workspace, unsigned long long workspace_bytes, void* stream);

/* Scratch bytes fa_bwd needs for these sizes (8 * B * H * N rounded up to 128 per head). */
int fa_bwd_workspace_size(int B, int H, int N, int d, unsigned long long* bytes);

/*
 * Standard attention with the N x N score matrix materialised in HBM: the comparison the
 * concept card "FlashAttention 2 + 3 — speicherbewusste Attention-Kernels" draws
 * ("Worum es geht": scores written to HBM and read back for the softmax and the
 * weighted sum; "Begriffe auf dieser Seite", HBM: 5-10 HBM passes against about one;
 * "Warum es zählt": 3-10x the GPU hours at long context).  Same operation, arguments and
 * outputs as fa_fwd, computed in three passes:
 *   1. S = scale * Q K^T in fp32 into the workspace (a cuBLAS strided-batched GEMM);
 *   2. a row softmax kernel: reads each row's visible scores once, writes P = softmax(S)
 *      in `dtype` over the start of the same row (zeros at masked columns), and the LSE;
 *   3. O = P V (a second cuBLAS GEMM), fp32 accumulation, rounded to `dtype`.
 *   workspace : device scratch of at least fa_fwd_naive_workspace_size() bytes, 256-byte
 *               aligned, owned by the caller: the fp32 scores (B * H * N * ceil(N/4)*4 * 4
 *               bytes, rounded up to 256) and then 32 MiB of scratch for the two GEMMs;
 *               calls sharing one workspace must not overlap on the GPU
 * Supported: fa_fwd's shapes with N <= 32768 and B*H*N < 2^31 (else FA_ERR_UNSUPPORTED or
 * FA_ERR_SHAPE).  cuBLAS (libcublas.so.13) is resolved at the first call, from the copy
 * the process already has loaded or from the loader's search path, and one cuBLAS handle
 * is created per device; each call points that handle at its own stream and at the GEMM
 * scratch in its own workspace, so calls with separate workspaces may overlap on separate
 * streams.  Calls from several host threads are serialised while they enqueue.
 * Errors as fa_fwd, plus FA_ERR_WORKSPACE, and FA_ERR_CUDA when cuBLAS cannot be loaded or
 * its handle created.
 */
int fa_fwd_naive(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, int dtype, void* workspace, unsigned long long workspace_bytes,
                 void* stream);

/* Scratch bytes fa_fwd_naive needs: the fp32 score matrix of every head, then 32 MiB for the GEMMs. */
int fa_fwd_naive_workspace_size(int B, int H, int N, int d, unsigned long long* bytes);

/* Size of the static scratch area behind fa_decode_noalloc, per device (8 MiB). */
#define FA_DECODE_NOALLOC_SCRATCH_BYTES (8ull << 20)

/*
 * fa_decode without a workspace argument, for callers that cannot allocate
 * device memory: a plugin that the host program hands only its input and output
 * buffers, or a serving loop that must not allocate once it has started.  The
 * attention pages define no such call; it computes exactly what fa_decode
 * computes, with the same arguments (minus workspace), the same kernels and the
 * same results.
 *
 * The split scratch is a fixed FA_DECODE_NOALLOC_SCRATCH_BYTES array of device
 * memory inside this library (one per device, reserved when the library's device
 * code is loaded there).  The call allocates nothing: no cudaMalloc, no pool, no
 * allocating library routine.
 *   - Limit: with num_splits = 0 fa_decode never picks a split count that needs
 *     more than 4 MiB of scratch, so only an explicit large num_splits can exceed
 *     the area.  When fa_decode_workspace_size reports more
 *     than FA_DECODE_NOALLOC_SCRATCH_BYTES for these sizes, the call returns
 *     FA_ERR_WORKSPACE and launches nothing; use a smaller num_splits, or
 *     fa_decode with a workspace of your own.
 *   - Set-up: the first call on each device looks up the array's address with
 *     cudaGetSymbolAddress (which may load this library's device code on that
 *     device) and returns FA_ERR_CUDA if that fails.  Make that first call
 *     outside any stream capture.
 *   - Zeroing: none needed.  Each call writes every scratch slot it reads, before
 *     reading it.
 *   - Races: all calls on one device share the one array.  Calls that can run on
 *     the GPU at the same time (on two streams, or from two host threads without
 *     ordering) corrupt each other's results; keep them on one stream or order
 *     them with events.
 * Other errors are those of fa_decode.
 */
int fa_decode_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                      int Nq, int Nk, int d, float scale, int causal, int dtype, int num_splits,
                      void* stream);

/* Static English text for a status code (never NULL). */
const char* fa_strerror(int status);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word, which kernels set when a bounded pipeline wait gives up.  Returns FA_OK
 * or FA_ERR_DEVICE_TIMEOUT; *bits (if not NULL) receives the raw word
 * (1 load warp, or a quantisation load wait; 2 MMA warp; 4 softmax warps; 8 drain
 * of in-flight copies; 16 a decode load wait).
 */
int fa_last_device_status(void* stream, unsigned int* bits);

/*
 * Test hook for the failure path: the next fa_fwd call's producer leaves out
 * the K/V loads of the pipeline step that holds K/V load number `load_index`
 * of every CTA (so the consumers' bounded waits run out), and every wait of
 * that call gives up after `timeout_ms` ms.  The
 * call still returns FA_OK; fa_last_device_status then reports the timeout.
 * load_index < 0 clears the hook.  Not for production use.
 */
int fa_debug_inject_stall(int load_index, int timeout_ms);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int fa_version(void);

/* Identity of the sources this library was compiled from: 16 hex digits of a SHA-256
 * over the CUDA sources, this header, the build script and the compiler flags
 * ("unknown" if built without the build script).  Static storage, never NULL. */
const char* fa_build_id(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H_ */
