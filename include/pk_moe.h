/*
 * pk_moe.h -- C ABI of the GB300 (sm_103a) MoE token-dispatch + expert-GEMM
 * library, libpkmoe.so.
 *
 * The operation is the single-device core of the expert-parallel
 * "token-dispatch + GEMM" of "Loads and Loads of Fluffy Kittens" (section
 * "Key claims", Fig. 17: top_k=8, num_experts=256, D=7168, D_expert=2048;
 * "Results", last item): tokens routed to experts are grouped expert by
 * expert, and each group is multiplied by its expert's up-projection weight.
 *
 * Tensors (all row-major, all in DEVICE memory, all owned and allocated by the
 * caller; the library allocates no device memory in any call):
 *   x              bf16  [T, D]            token activations
 *   topk_idx       int32 [T, k]            routed experts; slot s of token t
 *   W              bf16  [E, D, D_expert]  expert up-projection weights
 *   expert_counts  int32 [E]               rows routed to each expert
 *   expert_offsets int32 [E + 1]           exclusive prefix sum of the counts
 *   perm           int32 [T*k]             sorted row j -> flat index t*k+s
 *   inv_perm       int32 [T*k]             flat index t*k+s -> sorted row j
 *   out            bf16  [T*k, D_expert]   row j = x[perm[j] / k] @ W[e(j)]
 * bf16 tensors are passed as uint16_t bit patterns.
 *
 * Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is
 * the legacy default stream) and do not synchronise. route_counts ->
 * build_perm -> dispatch_gemm must be ordered on one stream (or by events).
 * Calls on distinct streams with distinct buffers are thread safe. The
 * routing kernels are launched with programmatic stream serialisation: one
 * may be scheduled while the kernel ahead of it in the stream is finishing,
 * but it waits for that kernel to complete before its first read or write of
 * global memory, so stream order holds for every buffer (also under CUDA
 * graph capture).
 *
 * Return value: PK_OK, or the first synchronous failure -- argument checks
 * (PK_ERR_INVALID_ARG, PK_ERR_UNSUPPORTED) or a failed launch (PK_ERR_CUDA).
 * Errors found on the device are written to *status_word (int32, device
 * memory, nullable): the first error code sticks until the caller clears it.
 * PK_ERR_BAD_INDEX means an expert index outside [0, E) (that entry is left
 * out of counts and perm, so outputs are incomplete); PK_ERR_TIMEOUT means a
 * bounded pipeline wait inside the GEMM ran out (outputs incomplete, the
 * kernel returned normally and the context stays usable).
 */
#ifndef PK_MOE_H
#define PK_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PK_OK = 0,
    PK_ERR_INVALID_ARG = 1,
    PK_ERR_UNSUPPORTED = 2,
    PK_ERR_CUDA = 3,
    PK_ERR_TIMEOUT = 4,
    PK_ERR_BAD_INDEX = 5,
    PK_ERR_CAPTURE = 6
} pk_status;

/* Largest number of experts the routing kernels accept. */
#define PK_MAX_EXPERTS 4096

/* Static string naming a status code (never NULL). */
const char* pk_status_str(int status);

/* Version of this ABI (major * 10000 + minor * 100 + patch). 1.1: FP8
 * entry points (quantisation, dispatch and grouped GEMM), GEMM kernel
 * selection, routing launch count. 1.2: PK_ERR_CAPTURE, the GEMM stall test
 * hook, MXFP8 quantisation and dispatch GEMM. */
#define PK_ABI_VERSION 10200
int pk_abi_version(void);

/*
 * Bytes of device workspace that pk_moe_route_counts and pk_moe_build_perm
 * need for (T, k, E): per-block expert histograms that become per-block
 * starting positions. 0 when T*k == 0. Pure host arithmetic.
 */
size_t pk_moe_workspace_bytes(int32_t T, int32_t k, int32_t E);

/*
 * Routing histogram and exclusive scan ("route tokens to experts", the
 * dispatch half of the token-dispatch + GEMM result, "Key claims", Fig. 17):
 *   expert_counts[e]    = #{(t, s) : topk_idx[t, s] == e}
 *   expert_offsets[0]   = 0,  expert_offsets[e+1] = expert_offsets[e] + expert_counts[e]
 * so expert_offsets[E] == T*k when every index is in range.
 *   topk_idx        device int32 [T, k], read only
 *   expert_counts   device int32 [E], written; may be NULL
 *   expert_offsets  device int32 [E + 1], written
 *   workspace       device, >= pk_moe_workspace_bytes(T, k, E) bytes, 16-byte
 *                   aligned; written here and read by pk_moe_build_perm
 *   status_word     device int32, nullable (see above)
 * Requires T >= 0, 1 <= k <= E <= PK_MAX_EXPERTS, T*k < 2^31. T == 0 writes
 * zero offsets.
 */
int pk_moe_route_counts(const int32_t* topk_idx, int32_t T, int32_t k, int32_t E,
                        int32_t* expert_counts, int32_t* expert_offsets,
                        void* workspace, size_t workspace_bytes,
                        int32_t* status_word, void* stream);

/*
 * Stable permutation of the routed rows, ordered by expert, then token, then
 * slot: for every flat index f = t*k + s with e = topk_idx[t, s],
 *   perm[expert_offsets[e] + r] = f,   inv_perm[f] = expert_offsets[e] + r,
 * where r = #{f' < f : topk_idx.flat[f'] == e}.
 *   topk_idx, expert_offsets  device int32, read only (offsets from
 *                   pk_moe_route_counts on the same topk_idx)
 *   perm            device int32 [T*k], written
 *   inv_perm        device int32 [T*k], written; may be NULL
 *   workspace       the workspace that pk_moe_route_counts filled for the same
 *                   topk_idx, T, k, E, unmodified since
 * Positions outside [0, T*k) (a workspace that does not match) are never
 * written; they set PK_ERR_BAD_INDEX.
 */
int pk_moe_build_perm(const int32_t* topk_idx, int32_t T, int32_t k, int32_t E,
                      const int32_t* expert_offsets, int32_t* perm, int32_t* inv_perm,
                      const void* workspace, size_t workspace_bytes,
                      int32_t* status_word, void* stream);

/*
 * Token dispatch fused with the expert GEMM ("token-dispatch + GEMM", "Key
 * claims", Fig. 17): for every expert e and sorted row j in
 * [expert_offsets[e], expert_offsets[e+1]),
 *   out[j, n] = bf16_rne( sum_d x[perm[j] / k, d] * W[e, d, n] )
 * with bf16 products accumulated in fp32 on the tensor cores. The gathered
 * rows are never written to memory: they are gathered from x straight into
 * shared memory. Experts with no rows cost nothing and their W is not read.
 *   x        device bf16 [T, D], 16-byte aligned
 *   perm     device int32 [T*k]; expert_offsets device int32 [E + 1]
 *   W        device bf16 [E, D, D_expert], 16-byte aligned
 *   out      device bf16 [T*k, D_expert], 16-byte aligned; rows of each expert
 *            segment written, nothing else
 * Requires T >= 0, k >= 1, E >= 1, D >= 1, D_expert >= 1, D and D_expert
 * multiples of 8, T*k < 2^31. Offsets are clamped into [0, T*k] and perm
 * entries into range, so no input makes the kernel touch memory outside the
 * buffers above; a perm entry outside [0, T*k) sets PK_ERR_BAD_INDEX.
 */
int pk_moe_dispatch_gemm(const uint16_t* x, const int32_t* perm, const int32_t* expert_offsets,
                         const uint16_t* W, int32_t T, int32_t k, int32_t D, int32_t E,
                         int32_t D_expert, uint16_t* out, int32_t* status_word, void* stream);

/*
 * FP8 variant of the dispatch GEMM ("ThunderKittens 2.0 & FP8/NVFP4": FP8
 * tensor-core primitives on Blackwell; the pages fix no scaling granularity,
 * so this takes one fp32 scale per token row of x and one per output column
 * of each W_e). With codes from pk_moe_quant_rows / pk_moe_quant_weights:
 *   out[j, n] = bf16_rne( (sum_d E4M3(xq[t, d]) * E4M3(wq[e, n, d])) * sx[t] * sw[e, n] )
 *   for t = perm[j] / k, j in expert e's segment; the sum runs on the tensor
 *   cores (tcgen05.mma kind::f8f6f4) with fp32 accumulation, the two scale
 *   multiplications in fp32, in that order.
 *   xq       device uint8 E4M3 codes [T, D], 16-byte aligned
 *   sx       device fp32 [T]
 *   perm     device int32 [T*k]; expert_offsets device int32 [E + 1]
 *   wq       device uint8 E4M3 codes of W in the blocked layout written by
 *            pk_moe_quant_weights (pk_moe_fp8_weight_bytes bytes), 16-byte
 *            aligned
 *   sw       device fp32 [E, D_expert], 16-byte aligned
 *   out      device bf16 [T*k, D_expert], 16-byte aligned
 * Requires D a multiple of 16, D_expert a multiple of 8,
 * pk_moe_fp8_weight_bytes(E, D, D_expert) < 2^38; otherwise as
 * pk_moe_dispatch_gemm (clamped offsets, PK_ERR_BAD_INDEX for a perm entry
 * outside [0, T*k), whose row then gets scale 0).
 */
int pk_moe_dispatch_gemm_fp8(const uint8_t* xq, const float* sx, const int32_t* perm,
                             const int32_t* expert_offsets, const uint8_t* wq, const float* sw,
                             int32_t T, int32_t k, int32_t D, int32_t E, int32_t D_expert,
                             uint16_t* out, int32_t* status_word, void* stream);

/*
 * E4M3 quantisation of the activations, one fp32 scale per row: with
 * a = max_d |x[t, d]| (bf16 values),
 *   sx[t]     = a / 448                      (1 if a == 0)
 *   xq[t, d]  = E4M3_rne_satfinite(x[t, d] * (448 / a))   (x[t, d] * 1 if a == 0)
 * every operation in IEEE fp32 with round-to-nearest-even, so the codes are
 * a pure function of x. 448 is the largest finite E4M3 value.
 *   x   device bf16 [T, D], 16-byte aligned; xq device uint8 [T, D], 8-byte
 *   aligned; sx device fp32 [T]. Requires D a multiple of 8.
 */
int pk_moe_quant_rows(const uint16_t* x, int32_t T, int32_t D, uint8_t* xq, float* sx,
                      void* stream);

/*
 * E4M3 quantisation of the expert weights, one fp32 scale per (expert,
 * output column), for the FP8 GEMM: with a = max_d |W[e, d, n]|,
 *   sw[e, n]        = a / 448                (1 if a == 0)
 *   code(e, n, d)   = E4M3_rne_satfinite(W[e, d, n] * (448 / a))
 * in IEEE fp32 as above. Done once per weight set. The codes are stored in
 * a blocked layout of 64-column x 128-code blocks, each 8 KiB block
 * contiguous so that the GEMM reads it from memory in one piece:
 *   wq[(((e * NB + n / 64) * KB + d / 128) * 64 + n % 64) * 128 + d % 128]
 *     = code(e, n, d),  NB = ceil(N / 64), KB = ceil(D / 128),
 * and every byte of a block past N or D is 0.
 *   W   device bf16 [E, D, N], 16-byte aligned; wq device uint8,
 *   pk_moe_fp8_weight_bytes(E, D, N) bytes, 16-byte aligned; sw device fp32
 *   [E, N], 4-byte aligned. A misaligned pointer returns PK_ERR_INVALID_ARG
 *   before any CUDA call.
 */
size_t pk_moe_fp8_weight_bytes(int32_t E, int32_t D, int32_t N);
int pk_moe_quant_weights(const uint16_t* W, int32_t E, int32_t D, int32_t N, uint8_t* wq,
                         float* sw, void* stream);

/*
 * Microscaled FP8 (MXFP8) form of the expert GEMM: the "Microscaling FP8"
 * tensor-core primitive named by the "ThunderKittens 2.0 & FP8/NVFP4" item of
 * the ThunderKittens tutorial page; the format follows the definition of the
 * MX formats. Along D, every 32 consecutive elements share one power-of-two
 * scale 2^s stored as an E8M0 byte s + 127, with
 *   s = floor(log2(max |v|)) - 8 (clamped to [-127, 127]; -127 for an
 *       all-zero block),  code = E4M3_rne_satfinite(v * 2^-s)  (in fp32).
 *
 * pk_moe_quant_rows_mx: x device bf16 [T, D], D a multiple of 32, 16-byte
 *   aligned -> xq device uint8 [T, D] codes (16-byte aligned) and sx device
 *   uint8 [T, D / 32] scale bytes (block b of row t covers d in [32 b, 32 b+32)).
 * pk_moe_quant_weights_mx: W device bf16 [E, D, N], D a multiple of 128, N a
 *   multiple of 8, all pointers 16-byte aligned -> wq: codes of the columns of
 *   every W[e] in the blocked layout of pk_moe_quant_weights
 *   (pk_moe_fp8_weight_bytes(E, D, N) bytes); swb: the blocks' scale bytes,
 *   pk_moe_mx_weight_scale_bytes(E, D, N) bytes, laid out for the GEMM: one
 *   1 KiB piece per (expert e, tile of 192 columns t, group of 128 d ks) at
 *   ((e * ceil(N / 192) + t) * (D / 128) + ks) * 1024; in it, bytes
 *   h * 512 + r * 16 + g * 4 + j hold the scale of block 4 ks + j of column
 *   192 t + 128 h + 32 g + r (h < 2, r < 32, g < 4); other bytes are zero.
 * pk_moe_dispatch_gemm_mxfp8: for every expert e and sorted row j in
 *   [expert_offsets[e], expert_offsets[e+1]),
 *     out[j, n] = bf16_rne( sum_d (q(x)[t, d] * 2^sx[t, d/32])
 *                                * (q(W)[e, d, n] * 2^sw[e, n, d/32]) ),
 *   t = perm[j] / k, on block-scaled tensor-core MMAs with fp32 accumulation.
 *   xq, wq, swb from the two calls above (xq, wq, swb, out 16-byte aligned,
 *   sx 4-byte aligned); D a multiple of 128, D_expert of 8. Otherwise as
 *   pk_moe_dispatch_gemm (clamped offsets, PK_ERR_BAD_INDEX for a perm entry
 *   outside [0, T*k)). Always the one-CTA kernel.
 */
int pk_moe_quant_rows_mx(const uint16_t* x, int32_t T, int32_t D, uint8_t* xq, uint8_t* sx,
                         void* stream);
size_t pk_moe_mx_weight_scale_bytes(int32_t E, int32_t D, int32_t N);
int pk_moe_quant_weights_mx(const uint16_t* W, int32_t E, int32_t D, int32_t N, uint8_t* wq,
                            uint8_t* swb, void* stream);
int pk_moe_dispatch_gemm_mxfp8(const uint8_t* xq, const uint8_t* sx, const int32_t* perm,
                               const int32_t* expert_offsets, const uint8_t* wq,
                               const uint8_t* swb, int32_t T, int32_t k, int32_t D, int32_t E,
                               int32_t D_expert, uint16_t* out, int32_t* status_word,
                               void* stream);

/*
 * Grouped GEMM of rows already in expert order -- the expert MLP's
 * down-projection that follows the up-projection above (same expert
 * segments; "Key claims", Fig. 17 gives D=7168, D_expert=2048): for every
 * expert e and row j in [expert_offsets[e], expert_offsets[e+1]),
 *   out[j, n] = bf16_rne( sum_c A[j, c] * W[e, c, n] )
 * with fp32 accumulation on the tensor cores.
 *   A        device bf16 [R, K] (row j of expert segment e), 16-byte aligned
 *   W        device bf16 [E, K, N], 16-byte aligned
 *   out      device bf16 [R, N], 16-byte aligned; rows of each segment written
 * Requires K and N multiples of 8. Offsets are clamped into [0, R].
 */
int pk_moe_grouped_gemm(const uint16_t* A, const int32_t* expert_offsets, const uint16_t* W,
                        int32_t R, int32_t K, int32_t N, int32_t E, uint16_t* out,
                        int32_t* status_word, void* stream);

/*
 * FP8 variant of the grouped GEMM (E4M3 codes, as pk_moe_dispatch_gemm_fp8):
 *   out[j, n] = bf16_rne( (sum_c E4M3(Aq[j, c]) * E4M3(wq[e, n, c])) * sa[j] * sw[e, n] )
 * for every expert e and row j in [expert_offsets[e], expert_offsets[e+1]).
 *   Aq   device uint8 codes [R, K] (pk_moe_quant_rows of A), 16-byte aligned
 *   sa   device fp32 [R]
 *   wq   device uint8, blocked codes of W2 [E, K, N] from pk_moe_quant_weights, 16-byte aligned
 *   sw   device fp32 [E, N], 16-byte aligned
 *   out  device bf16 [R, N], 16-byte aligned; rows of each segment written
 * Requires K a multiple of 16, N a multiple of 8. Offsets are clamped into [0, R].
 */
int pk_moe_grouped_gemm_fp8(const uint8_t* Aq, const float* sa, const int32_t* expert_offsets,
                            const uint8_t* wq, const float* sw, int32_t R, int32_t K, int32_t N,
                            int32_t E, uint16_t* out, int32_t* status_word, void* stream);

/*
 * Router top-k (the selection the expert-parallel workload of "Key claims",
 * Fig. 17 describes with top_k=8 of num_experts=256; the pages leave the
 * router itself open): for every token t,
 *   topk_idx[t, s] = expert with the s-th largest logits[t, :] (equal logits
 *                    go to the lower expert index, so the k experts differ)
 *   gates[t, s]    = exp(l_s - l_0) / sum_s' exp(l_s' - l_0), l_s the
 *                    selected logits (softmax over the k selected)
 *   logits    device fp32 [T, E], read only (NaN logits are not supported)
 *   topk_idx  device int32 [T, k], written
 *   gates     device fp32 [T, k], written; may be NULL
 * Requires T >= 0, 1 <= k <= min(E, 32), E <= PK_ROUTER_MAX_EXPERTS.
 */
#define PK_ROUTER_MAX_EXPERTS 1024
int pk_moe_router_topk(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* topk_idx,
                       float* gates, void* stream);

/*
 * Combine: un-permute the expert outputs back to token order and weight them
 * (the step after the expert MLP in the expert-parallel token-dispatch +
 * GEMM, "Key claims", Fig. 17; the pages leave the gating open):
 *   y[t, c] = bf16_rne( sum_{s=0..k-1} gates[t, s] * src[inv_perm[t*k + s], c] )
 * with fp32 products and sum, s ascending.
 *   src       device bf16 [T*k, C] in expert-sorted row order, 16-byte aligned
 *   inv_perm  device int32 [T*k] from pk_moe_build_perm
 *   gates     device fp32 [T, k]; NULL means every gate is 1
 *   y         device bf16 [T, C], 16-byte aligned, written
 * Requires C a multiple of 8, T*k < 2^31. An inv_perm entry outside
 * [0, T*k) sets PK_ERR_BAD_INDEX and row 0 is read in its place.
 */
int pk_moe_combine(const uint16_t* src, const int32_t* inv_perm, const float* gates, int32_t T,
                   int32_t k, int32_t C, uint16_t* y, int32_t* status_word, void* stream);

/*
 * Routing without any device allocation (the pages have no counterpart: this
 * is an interface convenience, not a step of the method). Computes exactly
 * what pk_moe_route_counts followed by pk_moe_build_perm compute (counts,
 * offsets, perm, inv_perm), for callers that cannot call cudaMalloc -- a host
 * program that hands all device memory to its own pool at start-up, a plug-in
 * that may not bypass its host runtime's allocator, or a latency-critical path
 * that cannot afford cudaMalloc's implicit synchronisation -- and therefore
 * cannot provide a workspace.
 *   The per-chunk counters live in a fixed array of PK_NOALLOC_SCRATCH_BYTES
 * inside the library's device image, held by every GPU that loads the library
 * until the process exits. Sizes with ceil(T*k / 2048) * E * 4 bytes above
 * that limit are rejected with PK_ERR_UNSUPPORTED (E = 256 allows T*k up to
 * 2,097,152). The call allocates nothing and calls no cudaMalloc/cudaFree.
 *   The array's device address is looked up with the device current on the
 * first call in each CUDA context (and again when the current context is a
 * new one, e.g. after cudaDeviceReset), never during stream capture: a first
 * call in a context that is made while `stream` is being captured returns
 * PK_ERR_CAPTURE and launches nothing -- make one call before capturing. Every
 * call shares the one array and leaves its contents behind; each call rewrites
 * every counter it reads, so nothing needs clearing, but calls that overlap on
 * the GPU (other streams or host threads) race: order them on one stream.
 *   Arguments, layouts and status reporting as for pk_moe_route_counts and
 * pk_moe_build_perm (expert_counts and inv_perm may be NULL).
 */
#define PK_NOALLOC_SCRATCH_BYTES (1u << 20)
int pk_moe_route_noalloc(const int32_t* topk_idx, int32_t T, int32_t k, int32_t E,
                         int32_t* expert_counts, int32_t* expert_offsets, int32_t* perm,
                         int32_t* inv_perm, int32_t* status_word, void* stream);

/*
 * Number of kernels that pk_moe_route_counts followed by pk_moe_build_perm
 * launch for these sizes (host arithmetic, no CUDA call): 2 when T*k is at
 * most 4096 (counts and scan in one kernel, then the permutation), else 3
 * (histogram, scan, permutation). -1 for invalid sizes.
 */
int pk_moe_route_kernel_launches(int32_t T, int32_t k, int32_t E);

/*
 * Kernel used by pk_moe_dispatch_gemm and pk_moe_dispatch_gemm_fp8 for
 * later calls from this process (both compute the same result, within
 * fp32 summation order):
 *   PK_GEMM_KERNEL_AUTO    default: the one-CTA kernel (the faster on GB300)
 *   PK_GEMM_KERNEL_SINGLE  one CTA per SM, tcgen05.mma.cta_group::1 (M = 128)
 *   PK_GEMM_KERNEL_PAIR    2-CTA clusters, tcgen05.mma.cta_group::2 (M = 256):
 *                          each SM loads its own rows and half of each W tile;
 *                          fewer bytes per SM, but a cross-SM handshake on
 *                          every K-step makes it slower (ep: 2.21 vs 1.79 ms)
 * Returns PK_ERR_INVALID_ARG for any other value.
 */
#define PK_GEMM_KERNEL_AUTO 0
#define PK_GEMM_KERNEL_SINGLE 1
#define PK_GEMM_KERNEL_PAIR 2
int pk_moe_set_gemm_kernel(int kernel);

/*
 * Limit, in nanoseconds, on every pipeline wait inside the GEMM kernel
 * (default 4e9). A wait that runs out sets PK_ERR_TIMEOUT and the kernel
 * drains its own copies and returns. Applies to later launches from this
 * process. 0 restores the default.
 */
void pk_moe_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Failure-detection check of the bounded wait used by the GEMM pipeline: one
 * block waits on a shared-memory barrier that nothing ever completes, gives
 * up after `limit_ns` and writes PK_ERR_TIMEOUT to *status_word (device
 * int32). Returns PK_OK if the launch succeeded.
 */
int pk_debug_bounded_wait(int32_t* status_word, uint64_t limit_ns, void* stream);

/*
 * Failure-detection check of the GEMM pipeline itself (off by default). While
 * set, every launch of the one-CTA dispatch or grouped GEMM kernel has CTA
 * `cta` arm K-step `kstep` of its own sequence (its units in order, nk K-steps
 * each) without issuing that K-step's weight (and grouped-GEMM row) copies, so
 * the K-step's full barrier never completes: the MMA thread's bounded wait
 * runs out, writes PK_ERR_TIMEOUT to the status word and raises the CTA's
 * abort flag, every role leaves its loop (each waits for the copies it has in
 * flight, the MMA thread for its issued MMAs), TMEM is freed and the kernel
 * returns. Outputs of that launch are undefined. cta < 0 or kstep < 0 turns
 * it off. Not thread-safe with concurrent launches; meant for tests, together
 * with a short pk_moe_set_wait_limit_ns.
 */
void pk_debug_stall_gemm(int32_t cta, int64_t kstep);

#ifdef __cplusplus
}
#endif

#endif /* PK_MOE_H */
