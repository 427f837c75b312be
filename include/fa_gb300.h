/*
 * fa_gb300.h -- C ABI of the exact attention forward for NVIDIA GB300 (sm_103a).
 *
 * The operation is the exact attention forward of FlashAttention: for every
 * batch b and head h,
 *
 *     S = scale * Q K^T               (masked: key j > query i set to -inf when causal)
 *     P = softmax(S) by rows,         O = P V,
 *     LSE_i = ln sum_j exp(S_ij)      (natural log, over the unmasked j)
 *
 * as defined on the zzszmyf.github.io notes page "FlashAttention 原理是什么？
 * 为什么又省显存又快" (§2 the three-step definition, §5 online softmax, §6 the
 * per-row statistics kept for the backward recompute, §7.1 Algorithm 1) and on
 * the aiqz.cc "flash-attention-io-optimization" article (section 在线Softmax算法:
 * m_new, r = e^(m - m_new), l_new, O~_new, O = O~/l).  S and P never leave the
 * chip: K/V tiles are merged with a running row max m and a running exp-sum l,
 * so the result is exact up to floating-point rounding.  The per-row LSE is the
 * statistic a backward pass needs to rebuild P without storing it.
 *
 * Precision: bf16 inputs and output, fp32 accumulation of S and O, P rounded to
 * bf16 for the P V product, LSE in fp32.
 *
 * Threading: every entry point is reentrant.  Calls on different streams may
 * run concurrently.  The library keeps no per-call state and allocates no
 * device memory in fa_fwd; the only device-global state is the status word
 * read by fa_status().
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes: 0 on success, negative on error. */
#define FA_OK            0
#define FA_ERR_ARG      -1  /* a null or misaligned pointer, or an unsupported size        */
#define FA_ERR_ARCH     -2  /* the current device is not compute capability 10.3 (GB300)   */
#define FA_ERR_LAUNCH   -3  /* the CUDA launch (or the TMA descriptor encoding) failed     */
#define FA_ERR_TIMEOUT  -4  /* a device-side barrier wait gave up (see fa_status)           */
#define FA_ERR_CUDA     -5  /* another CUDA runtime call failed                             */
#define FA_ERR_WORKSPACE_TOO_LARGE -6  /* fa_fwd_gqa_static_workspace: the partials need more
                                          than FA_STATIC_WORKSPACE_BYTES                      */

/* Bits of the device status word (fa_status). */
#define FA_STATUS_TIMEOUT 0x1u  /* some CTA's bounded mbarrier wait expired and it bailed out */
#define FA_STATUS_V_RANGE 0x2u  /* fa_fwd / fa_fwd_gqa: a V tile outside the range the fp16 P V
                                   product can hold at the scale the call had reached (see
                                   fa_fwd); that call's O is not exact */

/*
 * fa_fwd -- exact attention forward, O and LSE.
 *
 * q, k, v : device pointers, bf16, contiguous [B, H, N, d] (row stride d).
 *           Read only.  Each must be 16-byte aligned.
 * o       : device pointer, bf16, contiguous [B, H, N, d].  Written.
 * lse     : device pointer, fp32, contiguous [B, H, N].  Written.
 *           o and lse must not overlap q, k, v or each other.
 * B, H, N : batch, heads, sequence length; each >= 1.  Any N is accepted
 *           (the last 128-row tile may be partial).  B*H*N <= 2^31 - 1.
 * d       : head dimension, 64 or 128.
 * scale   : multiplies Q K^T before the softmax (usually 1/sqrt(d)); finite.
 * causal  : nonzero masks key j for query i when j > i (square, top-left
 *           aligned: every row keeps at least key 0).
 * stream  : the CUDA stream the kernel is enqueued on (0 = legacy default).
 *
 * Ownership: the caller allocates every buffer; the call allocates nothing.
 * The call is asynchronous with respect to the host: it only enqueues one
 * kernel.  The arguments are validated before anything is enqueued; on an
 * error return nothing was written.  A device-side wait that gives up (never
 * expected in correct operation) does not surface here: it sets
 * FA_STATUS_TIMEOUT in the status word, which fa_status() reads.
 *
 * Precision: S, O and the row sums accumulate in fp32; P is rounded to fp16 for
 * the P V product, with V converted to fp16 in shared memory at a power-of-two
 * scale fixed per work item (a pair of 128-row query tiles over one key range) from
 * the first V tile it reads (1 unless that tile's largest |v| is below 2^-4 or at
 * least 65520).  A later V tile that fp16 cannot
 * hold at that scale (with the scale 1: any |v| >= 65520) is saturated and sets
 * FA_STATUS_V_RANGE; that call's O is then not exact.
 *
 * Returns FA_OK, FA_ERR_ARG, FA_ERR_ARCH or FA_ERR_LAUNCH.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, float scale, int causal, cudaStream_t stream);

/*
 * fa_fwd_gqa -- exact attention forward with grouped K/V heads, different query and
 * key lengths, and split-K/V (FlashDecoding) parallelism.
 *
 * Grouped-query attention (GQA; MQA when Hkv = 1) lets G = Hq / Hkv query heads share
 * one K/V head, so fewer K/V bytes are read (the aiqz.cc article, section 性能调优经验,
 * on MQA/GQA).  Query head h uses K/V head h / G.  Split-K/V is the FlashDecoding
 * scheme of the notes page, §12.1: the keys are cut into n_splits ranges computed in
 * parallel, each giving a partial (O_s, LSE_s), merged exactly by
 *     LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
 *
 * q       : device bf16 [B, Hq, Nq, d], contiguous.      Read only, 16-byte aligned.
 * k, v    : device bf16 [B, Hkv, Nk, d], contiguous.     Read only, 16-byte aligned.
 * o       : device bf16 [B, Hq, Nq, d].                  Written.
 * lse     : device fp32 [B, Hq, Nq].                     Written.
 * B, Hq, Hkv, Nq, Nk >= 1; Hq a multiple of Hkv; B*Hq*Nq and B*Hkv*Nk <= 2^31 - 1.
 * d       : 64 or 128.   scale > 0 and finite.
 * causal  : nonzero masks keys after each query's position, with the queries aligned
 *           to the END of the keys (query i sits at position Nk - Nq + i): decoding
 *           appends Nq new queries after Nk - Nq cached keys.  Nq = Nk is the square
 *           mask of fa_fwd.  A query that sees no key (only if Nq > Nk) gets O = 0 and
 *           LSE = -inf.
 * n_splits: 1..1024 key ranges.  1 writes O and LSE directly; more write fp32
 *           partials into the workspace and a second kernel merges them.
 * workspace, workspace_bytes: device scratch for n_splits > 1, 256-byte aligned, at
 *           least fa_fwd_gqa_workspace_bytes(B, Hq, Nq, d, n_splits) bytes, not
 *           overlapping any other argument; ignored (may be NULL) for n_splits = 1.
 *           Its contents on entry do not matter; it is clobbered.
 * stream  : CUDA stream; one or two kernels are enqueued, nothing is synchronised.
 *
 * Ownership, validation and errors as for fa_fwd.  fa_fwd(q,k,v,o,lse,B,H,N,...) is
 * fa_fwd_gqa with Hq = Hkv = H, Nq = Nk = N, n_splits = 1.
 */
int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
               int n_splits, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes fa_fwd_gqa needs for these sizes (0 for n_splits = 1 or bad sizes). */
size_t fa_fwd_gqa_workspace_bytes(int B, int Hq, int Nq, int d, int n_splits);

/*
 * fa_fwd_gqa_static_workspace -- fa_fwd_gqa for callers that cannot allocate device
 * memory.  (An addition of this library; the FlashAttention pages have no counterpart.)
 *
 * Some callers cannot call cudaMalloc at the point where they run attention: a
 * serving loop that fixed its device-memory plan at start-up and may not allocate
 * afterwards, or a plain C host program that has no device allocator of its own to
 * hand out a scratch buffer.  This entry point takes the same arguments as
 * fa_fwd_gqa minus the workspace, and uses instead a workspace array of
 * FA_STATIC_WORKSPACE_BYTES (16 MiB) that the library defines in device memory.
 * Every GPU that loads the library holds that array until the process exits.
 *
 * It allocates nothing: no cudaMalloc, cudaFree or allocating library routine.  The
 * first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before any
 * stream capture.  Later calls reuse the address.
 *
 * All calls on a device share the one array, and it keeps whatever the last call
 * left there (the kernels overwrite every byte they read, so nothing needs
 * clearing).  Two calls whose kernels overlap on the GPU -- on different streams,
 * say -- race on the array and corrupt each other's results: serialise them.
 *
 * n_splits = 1 needs no workspace and behaves exactly as fa_fwd_gqa.  If the split
 * partials would need more than FA_STATIC_WORKSPACE_BYTES
 * (fa_fwd_gqa_workspace_bytes(B, Hq, Nq, d, n_splits) bytes), the call returns
 * FA_ERR_WORKSPACE_TOO_LARGE and enqueues nothing.  Other arguments and errors as for
 * fa_fwd_gqa.
 */
#define FA_STATIC_WORKSPACE_BYTES (16u << 20)
int fa_fwd_gqa_static_workspace(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                                int causal, int n_splits, cudaStream_t stream);

/*
 * fa_fwd_host -- fa_fwd_gqa (n_splits = 1) from host inputs to host outputs, with the
 * copies overlapped with the attention.  (An addition of this library: the pages'
 * IO-aware scheduling stops at HBM; this carries the same idea to the host link.)
 *
 * The K/V groups (b, hkv) are cut into chunks of groups_per_chunk groups (at most 64
 * chunks).  groups_per_chunk = 0 picks a default: when the copies take longer than the
 * attention (estimated at about 200 GB/s per direction and 1.3 PFLOP/s), at most seven
 * chunks of decreasing size (a quarter of the groups first, one thirty-second last);
 * otherwise eight equal chunks.  Chunk c's Q, K and V rows are copied host to
 * device on a copy stream of the library's; its forward runs, as soon as they have
 * landed, on one of two compute streams of the library's (alternating, so consecutive
 * chunks share the SMs); and its O and LSE rows go back on a second copy stream while
 * later chunks load and run.  Host-to-device copies, the kernels and device-to-host
 * copies of different chunks therefore overlap.  A chunk's kernel is the same as
 * fa_fwd_gqa's on those groups, so the results are bitwise those of fa_fwd_gqa.
 *
 * q_host, k_host, v_host : page-locked host memory (cudaHostAlloc / cudaMallocHost /
 *                  cudaHostRegister), the layouts of fa_fwd_gqa's q, k, v.  Read.
 * o_host, lse_host : page-locked host memory, the layouts of o and lse.  Written.
 * q, k, v, o, lse : device buffers of the full tensors, as for fa_fwd_gqa; q, k and v
 *                  are written here (they receive the copies).
 * Other arguments as for fa_fwd_gqa with n_splits = 1.
 *
 * Ownership and ordering: the caller owns every buffer; the call allocates no memory.
 * The first call on a device creates the library's four streams and its events
 * (kept until exit).  The call's work starts after the work already enqueued on
 * `stream`, and `stream` waits for the call's last copy: synchronise `stream` before
 * reading o_host / lse_host or reusing any buffer.  Calls on a device are enqueued one
 * at a time (a mutex); their copies share the two streams.
 *
 * Returns FA_OK; FA_ERR_ARG for the arguments fa_fwd_gqa rejects, a null or pageable
 * host buffer, host outputs that overlap host inputs or each other, or a negative
 * groups_per_chunk; FA_ERR_ARCH; FA_ERR_LAUNCH; FA_ERR_CUDA if a stream, event or
 * copy call fails (work already enqueued then stays enqueued).
 */
int fa_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                float* lse_host, void* q, void* k, void* v, void* o, float* lse, int B, int Hq,
                int Hkv, int Nq, int Nk, int d, float scale, int causal, int groups_per_chunk,
                cudaStream_t stream);

/*
 * fa_fwd_fp8 -- attention forward with FP8 (E4M3) tensor-core products: block-wise
 * quantisation with incoherent processing (§10 item ③ and §12.2 of the zzszmyf.github.io
 * notes "FlashAttention 原理是什么？为什么又省显存又快").
 *
 * Q and K are rotated row by row, q' = (q * signs) H / sqrt(128) with H the 128 x 128
 * Hadamard matrix, which leaves every score q.k unchanged and spreads outlier coordinates.
 * Q', K' and V are then quantised per 128-row tile of each (batch, head) to E4M3 codes with
 * one fp32 scale per tile (max|x| / 448).  The scores come from E4M3 products with fp32
 * accumulation and the descales; P is rounded to E4M3 for its product with V.  O and LSE have
 * the meaning they have in fa_fwd (LSE from the unrounded P).
 *
 * q, k, v   : device, bf16, contiguous [B, H, N, 128].  Read only.  16-byte aligned.
 * signs     : device, int8 [128], 16-byte aligned; a negative entry means -1, any other +1.
 *             Read only.
 * o, lse    : device, bf16 [B, H, N, 128] and fp32 [B, H, N].  Written.
 * d         : must be 128.  N >= 1 and ceil(N / 128) <= 1024.  scale finite and > 0.
 * causal    : nonzero = query i sees keys 0..i.
 * workspace : device, 256-byte aligned, at least fa_fwd_fp8_workspace_bytes(B, H, N, d)
 *             bytes, with N_pad = 128 * ceil(N / 128) and T = N_pad / 128:
 *               [0, C)        Q' codes, E4M3 [B*H, N_pad, 128]
 *               [C, 2C)       K' codes, E4M3 [B*H, N_pad, 128]
 *               [2C, 3C)      V codes transposed, E4M3 [B*H, 128, N_pad]
 *               then three fp32 arrays [B*H, T] of tile scales (Q', K', V), each at a
 *               256-byte boundary;  C = B*H*N_pad*128 rounded up to 256.
 *             Rows past N hold zero codes.  The call writes it; it is left holding the
 *             quantised tensors.
 * No output may overlap an input or the workspace.  Two kernels are enqueued on `stream`;
 * on an error return nothing was enqueued.  A device-side wait that gives up sets
 * FA_STATUS_TIMEOUT.
 *
 * Returns FA_OK, FA_ERR_ARG, FA_ERR_ARCH or FA_ERR_LAUNCH.
 */
int fa_fwd_fp8(const void* q, const void* k, const void* v, const signed char* signs, void* o,
               float* lse, int B, int H, int N, int d, float scale, int causal, void* workspace,
               size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_fwd_fp8_host -- fa_fwd_fp8 from host inputs to host outputs, with the copies overlapped
 * with the kernels.  (An addition of this library, like fa_fwd_host.)
 *
 * The B*H heads are cut into chunks (groups_per_chunk heads each, at most 64 chunks; 0 picks
 * the default of fa_fwd_host, with the two kernels' time estimated at about 1.35 PFLOP/s).
 * Chunk c's rows of q, k and v are copied host to device on a copy stream of the library's,
 * fa_fwd_fp8's two kernels run on them on one of two compute streams, and the chunk's o and
 * lse rows go back on a second copy stream.  Each compute stream uses its own part of the
 * workspace, laid out for the largest chunk; when two parts do not fit in workspace_bytes all
 * chunks run on one compute stream.  The results are bitwise fa_fwd_fp8's; the workspace is
 * scratch (its contents after the call are not specified).
 *
 * q_host, k_host, v_host : page-locked host memory, bf16 [B, H, N, 128].  Read.
 * o_host, lse_host : page-locked host memory, the layouts of o and lse.  Written.
 * q, k, v, o, lse, signs, workspace : device buffers as for fa_fwd_fp8; q, k, v receive the
 *                  copies.
 * Other arguments, ownership, ordering and errors as for fa_fwd_fp8 and fa_fwd_host.
 */
int fa_fwd_fp8_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                    float* lse_host, void* q, void* k, void* v, const signed char* signs, void* o,
                    float* lse, int B, int H, int N, int d, float scale, int causal,
                    void* workspace, size_t workspace_bytes, int groups_per_chunk,
                    cudaStream_t stream);

/* Bytes of workspace fa_fwd_fp8 needs (0 for sizes it would reject: d != 128, B, H, N < 1). */
size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_bwd -- exact attention backward: dQ, dK, dV from the forward's O and LSE.
 *
 * The forward saves only O and the per-row LSE; this call rebuilds S = scale*Q K^T
 * and P = exp(S - LSE) on chip, tile by tile, instead of reading an N x N matrix
 * (§6 "Recomputation" of the zzszmyf.github.io notes "FlashAttention 原理是什么？
 * 为什么又省显存又快"; the backward item of the aiqz.cc article's 工程实现细节
 * section).  With D = rowsum(dO * O) it computes
 *     dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q,
 * summing dK and dV over the G = Hq / Hkv query heads that share a K/V head.
 *
 * q, o, dout : device, bf16, contiguous [B, Hq, N, d].  Read only.
 * k, v       : device, bf16, contiguous [B, Hkv, N, d].  Read only.
 * lse        : device, fp32, [B, Hq, N] -- the forward's LSE (natural log).  Read only.
 * dq         : device, bf16, [B, Hq, N, d].  Written.
 * dk, dv     : device, bf16, [B, Hkv, N, d].  Written.
 * delta      : device, fp32, [B, Hq, N].  Written with D = rowsum(dO * O) (fp32 sum of
 *              bf16 products); the call's scratch, left holding D on return.
 * Every pointer is 16-byte aligned; no output overlaps an input or another output.
 * B, Hq, Hkv, N >= 1 with Hq % Hkv == 0 (queries and keys have the same length N);
 * d is 64 or 128; scale finite and > 0; causal: nonzero = query i sees keys 0..i.
 * B*Hq*N <= 2^31 - 1.  Three kernels are enqueued on `stream` (D, then dK/dV, then
 * dQ); the call returns once they are enqueued.  The dQ kernel, which reads nothing the
 * dK/dV kernel writes, is launched as its programmatic dependent and may start before it
 * ends, but it completes only after it, so whatever the stream runs after this call sees
 * dQ, dK and dV complete.  On FA_ERR_ARG or FA_ERR_ARCH nothing was enqueued; on
 * FA_ERR_LAUNCH the kernels before the failing launch may have been.  A device-side wait
 * that gives up sets FA_STATUS_TIMEOUT (fa_status).
 *
 * Returns FA_OK, FA_ERR_ARG, FA_ERR_ARCH or FA_ERR_LAUNCH.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, float* delta, int B, int Hq, int Hkv,
           int N, int d, float scale, int causal, cudaStream_t stream);

/*
 * fa_bwd_host -- fa_bwd from host inputs to host outputs, with the copies overlapped with
 * the kernels.  (An addition of this library, like fa_fwd_host.)
 *
 * The K/V groups are cut into chunks (groups_per_chunk each, at most 64 chunks; 0 picks a
 * default as fa_fwd_host does, with the backward's time estimated at about 0.85 PFLOP/s).
 * Chunk c's rows of q, k, v, o, lse and dout are copied host to device on a copy stream of
 * the library's, fa_bwd's three kernels run on them on one of two compute streams, and the
 * chunk's dq, dk and dv rows go back on a second copy stream while later chunks load and run.
 * A chunk's kernels are fa_bwd's on those groups, so the results are bitwise fa_bwd's.
 *
 * q_host .. dout_host : page-locked host memory, the layouts of fa_bwd's inputs.  Read.
 * dq_host, dk_host, dv_host : page-locked host memory, the layouts of dq, dk, dv.  Written.
 * q .. dout, dq, dk, dv, delta : device buffers as for fa_bwd; the inputs receive the
 *                  copies; delta (D = rowsum(dO * O)) stays on the device.
 * Other arguments as for fa_bwd.
 *
 * Ownership, ordering and errors as for fa_fwd_host: the call allocates no memory, starts
 * after the work already on `stream`, and `stream` waits for its last copy.  FA_ERR_ARG also
 * for a null or pageable host buffer, host outputs that overlap host inputs or each other, or
 * a negative groups_per_chunk.
 */
int fa_bwd_host(const void* q_host, const void* k_host, const void* v_host, const void* o_host,
                const float* lse_host, const void* dout_host, void* dq_host, void* dk_host,
                void* dv_host, void* q, void* k, void* v, void* o, float* lse, void* dout, void* dq,
                void* dk, void* dv, float* delta, int B, int Hq, int Hkv, int N, int d, float scale,
                int causal, int groups_per_chunk, cudaStream_t stream);

/*
 * fa_status -- read the device status word of the current device.
 *
 * Synchronises `stream` first, then copies the word to the host.  If `clear`
 * is nonzero the word is reset to 0 afterwards.  Returns the word (>= 0) or
 * FA_ERR_CUDA.
 */
int fa_status(int clear, cudaStream_t stream);

/*
 * fa_fwd_withheld_tile -- test hook for the bounded device waits.
 *
 * Same arguments as fa_fwd, plus wait_timeout_ms.  The kernel's producer warp
 * deliberately never loads V tile 0, so the MMA warp's wait for it cannot be
 * satisfied; every wait in the kernel gives up after about wait_timeout_ms,
 * each CTA waits for the copies it has in flight, frees its tensor memory and
 * returns, and FA_STATUS_TIMEOUT is set.  No fault and no hang: the context
 * stays usable.  The contents of o and lse are unspecified afterwards.
 * wait_timeout_ms must lie in [1, 10000].
 */
int fa_fwd_withheld_tile(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int N, int d, float scale, int causal,
                         double wait_timeout_ms, cudaStream_t stream);

/*
 * fa_fwd_withheld_ring_tile -- the same test hook with the withheld tile chosen: ring_tile
 * (>= 0) indexes the K/V tiles of a CTA's first work item in the order its producer loads
 * them, K_0 = 0, V_0 = 1, K_1 = 2, V_1 = 3, ...  (fa_fwd_withheld_tile is ring_tile = 1).
 * CTAs whose first item loads fewer tiles run to completion; the others give up as above,
 * some after handing P over for the steps before the missing tile, and take on no further
 * item.  Returns FA_ERR_ARG for ring_tile < 0 or a timeout outside
 * [1, 10000] ms; otherwise as fa_fwd_withheld_tile.
 */
int fa_fwd_withheld_ring_tile(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int N, int d, float scale, int causal, int ring_tile,
                              double wait_timeout_ms, cudaStream_t stream);

/*
 * fa_bwd_withheld_tile, fa_fwd_fp8_withheld_tile -- the same test hook for the backward
 * and the FP8 forward.  Same arguments as fa_bwd / fa_fwd_fp8, plus wait_timeout_ms in
 * [1, 10000].  The backward's dK/dV producer never loads its first stage and its dQ
 * producer never loads V tile 0; the FP8 kernel's producer never loads V tile 0.  The
 * waits for them give up after about wait_timeout_ms, every CTA cleans up and returns,
 * and FA_STATUS_TIMEOUT is set; the outputs are unspecified afterwards.
 */
int fa_bwd_withheld_tile(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv,
                         float* delta, int B, int Hq, int Hkv, int N, int d, float scale,
                         int causal, double wait_timeout_ms, cudaStream_t stream);
int fa_fwd_fp8_withheld_tile(const void* q, const void* k, const void* v,
                             const signed char* signs, void* o, float* lse, int B, int H,
                             int N, int d, float scale, int causal, void* workspace,
                             size_t workspace_bytes, double wait_timeout_ms,
                             cudaStream_t stream);

/* fa_strerror -- a static, human-readable string for a return code. */
const char* fa_strerror(int code);

/* fa_version -- the library's interface version (currently 3). */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
