/*
 * nvfp4_skinny.h -- C ABI of the GB300 (sm_103a) NVFP4 W4A16 skinny decode library.
 *
 * What it computes (sources are the pages' titles and sections):
 *
 *   NVFP4 weight: w_hat[n,k] = e2m1(q[n,k]) * e4m3(s[n, k/16]) * g          (1)
 *     "E2M1 weights + E4M3 group-16 scales + FP32 global" -- gemma-cuda-hybrid
 *     README, "Everything it has / Inference engine"; the offline repack into
 *     MMA-fragment order -- same page, "Why it's NVIDIA-only ... /
 *     NVFP4-specific".
 *   Skinny GEMM: y[m,n] = sum_k w_hat[n,k] * x[m,k], M <= 16, fp32
 *     accumulate, bf16 in and out -- gemma-cuda-hybrid README, "Everything it
 *     has / Inference engine" (the tensor-core GEMM for all M<=16 GEMMs).
 *   MoE FFN: router top-k over the logits, softmax over the chosen k, grouped
 *     gate+up product, h = gelu_tanh(gate) * up, grouped down product,
 *     probability-weighted sum plus the always-on shared expert --
 *     TensorSharp docs/models/gemma4.md, "3.1 Per-layer (dense)", "3.2
 *     Per-layer (MoE)", "4.6 MoE", "14. Optimization opportunities / Completed
 *     (Expert-batched FFN)"; GELU-tanh -- TensorFold issue #1048, "Steps",
 *     step 2; "Grouped weight-resident MoE (no atomics ...)" -- gemma-cuda-hybrid
 *     README, "Everything it has / Inference engine".
 *   lm_head + greedy argmax: per token row the largest logit of W_hat . x and
 *     its lowest index, no logits written to memory -- gemma-cuda-hybrid
 *     README, "Headline numbers" (bit-exact greedy) and "Everything it has"
 *     (NVFP4 tied lm_head).
 *
 * Conventions for every call:
 *   - Pointers marked (device) are CUDA device pointers; (host) are host
 *     pointers.  The caller owns every buffer; the library allocates no memory
 *     on any call.
 *   - Device work is enqueued asynchronously on `stream` (0 = legacy default
 *     stream).  Arguments are checked on the host before anything is launched;
 *     a bad argument returns an error status and launches nothing.  A launch
 *     failure returns NVFP4_ERR_CUDA (the CUDA error is left for
 *     cudaGetLastError()).  No C++ exception crosses this boundary.
 *   - bf16 tensors are passed as uint16_t bit patterns, row-major, contiguous.
 *   - Preconditions not checked on the device: weights and activations are
 *     finite; router logits are finite or -inf (a NaN logit counts as -inf);
 *     expert ids passed to moe_ffn_grouped come from moe_route_topk;
 *     workspaces are not shared by calls that may run concurrently.
 *   - The weight-streaming calls launch with programmatic dependent launch:
 *     they start copying weights (data and global_scale) while the preceding
 *     kernel on the stream may still run, and read activations only after it
 *     has completed.  So a weight must be complete before the kernel just
 *     before the call starts, or be written by a kernel that does not use
 *     griddepcontrol.launch_dependents (nvfp4_quantize, nvfp4_repack and
 *     ordinary library or framework kernels do not).
 *   - Kernel waits are bounded (about one second); a wait that runs out sets a
 *     bit in a device error word read by nvfp4_device_error().
 */
#ifndef NVFP4_SKINNY_H_
#define NVFP4_SKINNY_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4_LAYOUT_VERSION 2u

/* Flags of an nvfp4_weight / nvfp4_repack call. */
#define NVFP4_GATED 1u /* rows are [gate (N/2) || up (N/2)], N % 64 == 0 */

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_NULL = 1,      /* a required pointer is NULL */
  NVFP4_ERR_SHAPE = 2,     /* a size is out of range or inconsistent */
  NVFP4_ERR_ALIGN = 3,     /* a pointer is not aligned as documented */
  NVFP4_ERR_WORKSPACE = 4, /* workspace NULL or smaller than *_workspace_bytes() */
  NVFP4_ERR_LAYOUT = 5,    /* nvfp4_weight.layout_version or flags mismatch */
  NVFP4_ERR_CUDA = 6       /* a CUDA launch or query failed */
} nvfp4_status;

/*
 * A repacked NVFP4 weight (a view; the caller owns the memory).
 *   data          (device) repacked bytes, nvfp4_repacked_bytes(n, k, num_matrices)
 *                 long, 16-byte aligned, written by nvfp4_repack().
 *   global_scale  (device) fp32 [num_matrices]: g of formula (1) per matrix.
 *   n, k          logical rows and columns of one matrix; k % 16 == 0.
 *   num_matrices  1, or E for a stack of E expert matrices [E, n, k].
 *   flags         NVFP4_GATED for a fused [gate || up] matrix, else 0;
 *                 must equal the flags given to nvfp4_repack().
 *   layout_version  NVFP4_LAYOUT_VERSION.
 *
 * Repacked layout (version 2): rows padded to a multiple of 64 and columns to a
 * multiple of 64 with zero bytes; a gated matrix (n % 64 == 0) first moves gate
 * row i to row 16*(i/8) + i%8 and up row i to 16*(i/8) + 8 + i%8.  The padded
 * matrix is cut into 576-byte tiles of 16 rows x 64 columns; tile (64-row group
 * G, 64-column chunk kc, 16-row block r) starts at byte 576*((G*KC + kc)*4 + r),
 * KC = padded columns / 64, so the four tiles of one group and chunk are 2,304
 * contiguous bytes.  In a tile, byte 16*lane + 4*kt + j (lane = 4*g + t) holds
 * columns c, c+1 of the tile's row g + 8*(j&1) with c = 64*kc + 16*kt + 2*t +
 * 8*(j>>1) (low nibble = column c), and byte 512 + 8*g + 2*kt + h holds the
 * scale of the tile's row g + 8*h, group 4*kc + kt: one 16-byte load per lane
 * gives an m16n8k16 A fragment for four 16-column groups.  Scale codes are
 * stored with their sign bit clear: a negative scale is folded into the signs
 * of its 16 elements.
 */
typedef struct {
  const void *data;
  const float *global_scale;
  int32_t n;
  int32_t k;
  int32_t num_matrices;
  uint32_t flags;
  uint32_t layout_version;
} nvfp4_weight;

/* Human-readable name of a status code (static string). */
const char *nvfp4_status_string(nvfp4_status st);

/* Library's repacked-layout version (NVFP4_LAYOUT_VERSION at build time). */
uint32_t nvfp4_layout_version(void);

/*
 * Device error word: bit 0 = a kernel's bounded wait ran out of time.  Reads
 * the word (synchronously, on the current device) into *out and clears it if
 * `clear` is nonzero.
 */
nvfp4_status nvfp4_device_error(uint32_t *out, int32_t clear);

/*
 * Self-test of the failure path of the bounded waits (no fault, no hang):
 * launches one CTA whose warps wait, with the kernels' own bounded
 * warp-collective wait, on an mbarrier phase that nothing completes, and give
 * up after limit_cycles SM clock cycles (1 .. 2^31) instead of the kernels'
 * ~1 s.  The kernel then sets bit 0 of the device error word and returns; the
 * context stays usable.  Asynchronous on `stream`; read the word with
 * nvfp4_device_error afterwards.  NVFP4_ERR_SHAPE for a limit out of range.
 */
nvfp4_status nvfp4_selftest_wait_timeout(int64_t limit_cycles, cudaStream_t stream);

/* Bytes of a repacked weight of num_matrices x [n, k] (0 for invalid sizes). */
size_t nvfp4_repacked_bytes(int32_t n, int32_t k, int32_t num_matrices);

/*
 * Offline quantizer (formula (1) in reverse):
 *   g = fp32(amax|W| / 2688) (one correctly rounded fp32 division); per
 *   16-group the scale is the E4M3 code nearest to the exact quotient
 *   bmax / (6 g), ties to even, saturating at 448; each element the E2M1 code
 *   nearest to the exact quotient w / (e4m3(scale) * g), ties to even,
 *   saturating at 6, with the sign of w kept; a group whose scale is 0 gets
 *   zero codes; an all-zero matrix gets g = 0.  (The quotients are float64
 *   divisions by exact divisors, which decide every code as the exact real
 *   quotient would.)
 *   w        (device) fp32 [num_matrices, n, k], k % 16 == 0.
 *   nibbles  (device) u8 [num_matrices, n, k/2], canonical: column 2i in the
 *            low nibble of byte i.
 *   scales   (device) u8 [num_matrices, n, k/16].
 *   global_scale (device) fp32 [num_matrices].
 *   ws       (device) nvfp4_quantize_workspace_bytes(num_matrices) bytes.
 */
size_t nvfp4_quantize_workspace_bytes(int32_t num_matrices);
nvfp4_status nvfp4_quantize(const float *w, int32_t num_matrices, int32_t n, int32_t k, uint8_t *nibbles,
                            uint8_t *scales, float *global_scale, void *ws, size_t ws_bytes,
                            cudaStream_t stream);

/*
 * Offline repack of canonical NVFP4 bytes into the kernel layout above.
 *   nibbles, scales (device) canonical, as written by nvfp4_quantize().
 *   out      (device) nvfp4_repacked_bytes(n, k, num_matrices) bytes, 16-byte
 *            aligned; every byte is written (padding with zeros).
 *   flags    0 or NVFP4_GATED (then n % 64 == 0).
 */
nvfp4_status nvfp4_repack(const uint8_t *nibbles, const uint8_t *scales, int32_t num_matrices, int32_t n,
                          int32_t k, uint32_t flags, void *out, cudaStream_t stream);

/*
 * The same repack on the host: canonical bytes in host memory to the kernel
 * layout in host memory (the caller copies it to the device).  Byte-identical
 * to nvfp4_repack() (both walk one index function).  Synchronous; needs no GPU.
 *   nibbles, scales (host) canonical, as above.
 *   out      (host) out_bytes >= nvfp4_repacked_bytes(n, k, num_matrices);
 *            every byte of the repacked size is written (padding with zeros).
 * Errors: NVFP4_ERR_NULL, NVFP4_ERR_SHAPE, NVFP4_ERR_LAYOUT (unknown flags),
 * NVFP4_ERR_WORKSPACE (out too small); nothing is written then.
 */
nvfp4_status nvfp4_repack_host(const uint8_t *nibbles, const uint8_t *scales, int32_t num_matrices, int32_t n,
                               int32_t k, uint32_t flags, void *out, size_t out_bytes);

/*
 * Dense skinny GEMM: y[m, :] = bf16( W_hat . x[m, :] ), 1 <= m <= 16.
 *   w   num_matrices == 1, flags == 0.
 *   x   (device) bf16 [m, w->k], 16-byte aligned.
 *   y   (device) bf16 [m, w->n], 4-byte aligned.
 *   ws  (device) nvfp4_gemm_workspace_bytes(m, n, k) bytes, 16-byte aligned.
 *       It holds the k-split fixup area: 512 KiB of arrival counters, then the
 *       partial sums.  The counters must be zero before the first call that
 *       uses this workspace (for example cudaMemsetAsync once after
 *       allocation); every completed call leaves them zero again, so the same
 *       workspace may serve calls of any shape whose size it covers.
 * M = 1 runs on CUDA cores (warp-shuffle reduction); M = 2..16 on m16n8k16
 * tensor-core MMAs with the weights as the 16-row operand and the tokens in one
 * (M <= 8) or two 8-slot columns.
 */
size_t nvfp4_gemm_workspace_bytes(int32_t m, int32_t n, int32_t k);
nvfp4_status nvfp4_gemm(const nvfp4_weight *w, const uint16_t *x, int32_t m, uint16_t *y, void *ws,
                        size_t ws_bytes, cudaStream_t stream);

/*
 * W4A4 NVFP4 (activations quantized too).  The pages do not describe this
 * variant; it follows the weights' recipe (gemma-cuda-hybrid README,
 * "Everything it has / Inference engine": E2M1 codes, E4M3 scales per 16
 * along K, an FP32 global scale), with one global scale per token row.
 *
 * nvfp4_quantize_act: bf16 activations -> NVFP4, each row quantized as a matrix
 * of its own (the codes and scales decided as in nvfp4_quantize), so a token's
 * codes do not depend on the rest of the batch.
 *   x             (device) bf16 [m, k], 1 <= m <= 4096, k % 16 == 0, 16-byte aligned.
 *   codes         (device) u8 [m, k/2] canonical (column 2i in the low nibble of
 *                 byte i), 8-byte aligned;  scales (device) u8 [m, k/16].
 *   global_scale  (device) fp32 [m]: amax of row m / 2688.
 *   ws            (device) nvfp4_quantize_workspace_bytes(m) bytes.
 *
 * nvfp4_gemm_w4a4 / lm_head_argmax_w4a4: nvfp4_gemm and lm_head_argmax with
 * the activations given as the output of nvfp4_quantize_act:
 *   y[m, n] = bf16( sum_k w_hat[n, k] * x_hat[m, k] ),
 *   x_hat[m, k] = e2m1(code) * e4m3(scale of k's 16-group) * global_scale[m].
 * x_codes 16-byte aligned, k = w->k.  The activations are dequantized into f16
 * tensor-core operands (exact) as the weights are; fp32 accumulation.
 * Workspaces and limits as nvfp4_gemm / lm_head_argmax (1 <= m <= 16).
 */
nvfp4_status nvfp4_quantize_act(const uint16_t *x, int32_t m, int32_t k, uint8_t *codes, uint8_t *scales,
                                float *global_scale, void *ws, size_t ws_bytes, cudaStream_t stream);
nvfp4_status nvfp4_gemm_w4a4(const nvfp4_weight *w, const uint8_t *x_codes, const uint8_t *x_scales,
                             const float *x_global, int32_t m, uint16_t *y, void *ws, size_t ws_bytes,
                             cudaStream_t stream);
nvfp4_status lm_head_argmax_w4a4(const nvfp4_weight *w, const uint8_t *x_codes, const uint8_t *x_scales,
                                 const float *x_global, int32_t m, float *max_logit, int32_t *argmax, void *ws,
                                 size_t ws_bytes, cudaStream_t stream);

/*
 * Router logits from the hidden state (TensorSharp docs/models/gemma4.md, "4.6
 * MoE", step 2: the router matmul, an unweighted RMSNorm, then the learned
 * per-expert scale ffn_gate_inp.scale):
 *   raw[m, e]    = W_hat . x_m  (the NVFP4 skinny GEMM, fp32 accumulate and output)
 *   logits[m, e] = raw[m, e] / sqrt(mean_e raw[m, e]^2 + eps) * gate_scale[e]
 * The result feeds moe_route_topk.
 *   w           the router weight, n = n_experts (<= 1024), k = hidden size;
 *               num_matrices == 1, flags == 0.
 *   x           (device) bf16 [m, w->k], 1 <= m <= 16, 16-byte aligned.
 *   gate_scale  (device) fp32 [n_experts], or NULL for all ones.
 *   eps         >= 0 (the pages give none; 1e-6 is the usual choice).
 *   logits      (device) fp32 [m, n_experts].
 *   ws          (device) nvfp4_gemm_workspace_bytes(m, n_experts, w->k) bytes,
 *               under the same rules as nvfp4_gemm's workspace.
 * Two launches on `stream` (the GEMM, then the normalisation).
 */
nvfp4_status moe_router_logits(const nvfp4_weight *w, const uint16_t *x, int32_t m, const float *gate_scale, float eps,
                               float *logits, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * MoE router: per token m, the top_k largest logits (descending; equal logits
 * -> lower expert id) and a softmax over those top_k logits; then a stable
 * grouping of the m*top_k (token, slot) pairs by expert with no atomics.
 *   logits          (device) fp32 [m, n_experts]
 *   ids             (device) int32 [m, top_k]
 *   probs           (device) fp32 [m, top_k]
 *   expert_offsets  (device) int32 [n_experts + 1]: expert e's pairs are
 *                   sorted_pairs[offsets[e] .. offsets[e+1]).
 *   sorted_pairs    (device) int32 [m * top_k]: pair index p = token*top_k + slot,
 *                   ascending within an expert.
 * Limits: 1 <= m <= 4096, 1 <= top_k <= 32, top_k <= n_experts <= 1024,
 * m * top_k <= 16384.
 * Logits: finite or -inf; a NaN counts as -inf.  Every id is a valid expert
 * (the top_k picks are distinct: -inf logits go to the lowest unchosen ids),
 * and a token whose logits are all -inf gets weight 0 on every slot.
 */
nvfp4_status moe_route_topk(const float *logits, int32_t m, int32_t n_experts, int32_t top_k, int32_t *ids,
                            float *probs, int32_t *expert_offsets, int32_t *sorted_pairs,
                            cudaStream_t stream);

/*
 * moe_route_topk with the routing-weight variants of TensorSharp
 * docs/models/gemma4.md: the same top_k ids and grouping, and
 *   flags & NVFP4_ROUTE_SOFTMAX_ALL: probs = the softmax over all n_experts
 *       logits read at the chosen experts (the literal topK(softmax(logits)) of
 *       "3.2 Per-layer (MoE)"; not renormalised, so a row sums to at most 1);
 *       otherwise the softmax over the top_k chosen logits.
 *   expert_scale (device) fp32 [n_experts] or NULL: each pair's weight times its
 *       expert's scale (a per-expert down-projection scale folded into the
 *       routing weights, "14. Optimization opportunities").
 * moe_ffn_grouped then applies these weights unchanged.  Other flag bits:
 * NVFP4_ERR_SHAPE.
 */
#define NVFP4_ROUTE_SOFTMAX_ALL 1
nvfp4_status moe_route_topk_ex(const float *logits, int32_t m, int32_t n_experts, int32_t top_k, int32_t flags,
                               const float *expert_scale, int32_t *ids, float *probs, int32_t *expert_offsets,
                               int32_t *sorted_pairs, cudaStream_t stream);

/*
 * Grouped MoE FFN: out[t] = bf16( sum_r probs[t,r] * down_e(h_{t,r}) + shared_down(h_{t,shared}) )
 * with h = bf16( gelu_tanh(gate_e . x_t) * (up_e . x_t) ) and e = ids[t, r].
 *   x               (device) bf16 [m, d], 16-byte aligned.
 *   probs, expert_offsets, sorted_pairs: as written by moe_route_topk.
 *   gate_up         stacked [E, 2*inter, d], flags NVFP4_GATED.
 *   down            stacked [E, d, inter], flags 0.
 *   shared_gate_up, shared_down: one matrix each of the same shapes, or both NULL.
 *   out             (device) bf16 [m, d].
 *   ws              (device) moe_ffn_workspace_bytes(m, top_k, E, d, inter) bytes,
 *                   16-byte aligned.  It holds a k-split fixup area (512 KiB of
 *                   arrival counters at its start, then partial sums), h and the
 *                   per-(token, slot) down outputs.  The counters must be zero
 *                   before the first call on this workspace (for example
 *                   cudaMemsetAsync once after allocation); every completed call
 *                   leaves them zero again, so one workspace of the largest size
 *                   needed serves calls of any shape.
 * Limits: 1 <= m <= 4096, m * top_k <= 16384, d % 64 == 0, inter % 64 == 0.
 * m > 16 is a prefill chunk: each expert's pairs (and the shared expert's
 * tokens) run in blocks of at most 32, each block's dequantized weight tiles
 * feeding four 8-slot tensor-core MMA columns.
 */
size_t moe_ffn_workspace_bytes(int32_t m, int32_t top_k, int32_t n_experts, int32_t d, int32_t inter);
nvfp4_status moe_ffn_grouped(const uint16_t *x, int32_t m, int32_t top_k, const float *probs,
                             const int32_t *expert_offsets, const int32_t *sorted_pairs,
                             const nvfp4_weight *gate_up, const nvfp4_weight *down,
                             const nvfp4_weight *shared_gate_up, const nvfp4_weight *shared_down,
                             uint16_t *out, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * One MoE layer in one call (gemma-cuda-hybrid README, "Everything it has /
 * Inference engine": the router's top-k, then the routed and shared experts'
 * SwiGLU FFNs, weighted and summed): moe_route_topk_ex (route_flags,
 * expert_scale as there) writing ids, probs, expert_offsets and sorted_pairs,
 * then moe_ffn_grouped on them, with the same results and workspace as the two
 * calls made in turn.  The number of experts is gate_up->num_matrices; logits is
 * [m, num_matrices] fp32.  All arguments of both steps are checked before the
 * first launch, so an error status means nothing was launched.
 */
nvfp4_status moe_forward(const uint16_t *x, const float *logits, int32_t m, int32_t top_k, int32_t route_flags,
                         const float *expert_scale, int32_t *ids, float *probs, int32_t *expert_offsets,
                         int32_t *sorted_pairs, const nvfp4_weight *gate_up, const nvfp4_weight *down,
                         const nvfp4_weight *shared_gate_up, const nvfp4_weight *shared_down, uint16_t *out, void *ws,
                         size_t ws_bytes, cudaStream_t stream);

/*
 * lm_head with fused greedy argmax: for each token row m, max_n (W_hat . x_m)[n]
 * in fp32 and the lowest n reaching it.  The vocabulary is split across CTAs
 * and K across the warps of a CTA; no logits are written to memory.
 *   w          num_matrices == 1, flags == 0 (n = vocabulary size).
 *   x          (device) bf16 [m, w->k], 1 <= m <= 16, 16-byte aligned.
 *   max_logit  (device) fp32 [m];  argmax (device) int32 [m].
 *   ws         (device) lm_head_workspace_bytes(m, n) bytes (4 KiB: an arrival
 *              counter and one packed (value, row) maximum per token), 16-byte
 *              aligned.  It must be zero before the first call on it (for
 *              example cudaMemsetAsync once after allocation); every completed
 *              call leaves it zero again.  The per-CTA maxima are combined with
 *              64-bit atomic maxima on (value, inverted row), so the result does
 *              not depend on the order the CTAs finish in.
 * A NaN logit counts as -inf, so the index is always a valid row: a token whose
 * logits are all NaN gets (-inf, 0).
 */
size_t lm_head_workspace_bytes(int32_t m, int32_t vocab);
nvfp4_status lm_head_argmax(const nvfp4_weight *w, const uint16_t *x, int32_t m, float *max_logit,
                            int32_t *argmax, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * lm_head with fused temperature sampling (Gumbel-max): for each token row m, the
 * n maximising (W_hat . x_m)[n] / temperature + g(n, m), with g standard Gumbel
 * noise, and that maximum -- a draw from softmax(logits / temperature); ties to
 * the lower n.  gemma-cuda-hybrid README, "Server": Gumbel-max temperature
 * sampling, temperature 0 reducing to exact greedy.  The noise is the
 * counter-based generator Philox4x32-10 (Salmon et al., SC 2011): word 0 of
 * Philox(counter (n, m, 0, 0), key (seed low 32 bits, seed high 32 bits)), u =
 * ((word >> 9) + 0.5) / 2^23, g = -log(-log u).  A call is deterministic in its
 * seed: pass a new seed for each step.  No logits or noise reach memory.
 *   temperature  > 0 samples; == 0 is lm_head_argmax (max_key = the max logit).
 *   max_key      (device) fp32 [m]: the winning logit / temperature + noise.
 *   token        (device) int32 [m].
 *   everything else as lm_head_argmax (same workspace).
 */
nvfp4_status lm_head_sample(const nvfp4_weight *w, const uint16_t *x, int32_t m, float temperature, uint64_t seed,
                            float *max_key, int32_t *token, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * lm_head_sample with the final-logit softcap of TensorSharp
 * docs/models/gemma4.md, "4.8 Logit softcap": every logit l becomes
 * softcap * tanh(l / softcap) before the temperature and the noise (softcap 0:
 * off, exactly lm_head_sample).  With temperature 0 this is the greedy argmax of
 * the capped logits, max_key being the capped maximum.  softcap must be finite
 * and >= 0 (else NVFP4_ERR_SHAPE); everything else as lm_head_sample.
 */
nvfp4_status lm_head_sample_ex(const nvfp4_weight *w, const uint16_t *x, int32_t m, float softcap, float temperature,
                               uint64_t seed, float *max_key, int32_t *token, void *ws, size_t ws_bytes,
                               cudaStream_t stream);

/*
 * lm_head_argmax without a caller-provided workspace.  The pages have no
 * counterpart to this call: it exists for callers that cannot allocate device
 * memory -- for example a plugin or runtime that hands the library only its
 * input and output buffers from a fixed pool, or a decode loop that must not
 * hit cudaMalloc's implicit device synchronisation or an out-of-memory failure
 * in the middle of a request.
 *
 * Same arguments, result and limits as lm_head_argmax, minus ws/ws_bytes.  The
 * scratch it needs (an arrival counter and the per-token packed maxima, 4,096
 * bytes) is a static array inside this library's device code, so every GPU that
 * loads the library holds it until the process exits.  No call allocates or
 * frees memory.
 *   - The first call on a device, with that device current, looks up the
 *     array's device address with cudaGetSymbolAddress and zeroes it
 *     (synchronously); make that first call before any stream capture.
 *   - Every call clears the arrival counter on `stream` before its kernel; the
 *     kernel's last CTA leaves the maxima zero for the next call.
 *   - All calls on a device share the one array: calls that may overlap on the
 *     GPU (other streams, other host threads) race and give wrong results.
 *     Serialise them, or use lm_head_argmax with separate workspaces.
 *   - Returns NVFP4_ERR_WORKSPACE if lm_head_workspace_bytes(m, w->n) exceeds
 *     the array (never for m <= 16).
 */
nvfp4_status lm_head_argmax_noalloc(const nvfp4_weight *w, const uint16_t *x, int32_t m, float *max_logit,
                                    int32_t *argmax, cudaStream_t stream);

/*
 * The launch plan a product would use, for host-side checks of the work
 * decomposition (no device work; no CUDA call).
 *   product  0 dense GEMM (n x k), 1 lm_head (n x k), 2 MoE gate+up (n = 2*inter,
 *            k = d), 3 MoE down (n = d, k = inter).
 *   m, top_k, n_experts  as the product's call (top_k, n_experts: MoE only).
 *   sms      the grid's SM count to plan for (the library plans for the device's).
 *   out      (host) int32 [10 or 11]: K split S, chunks per slice L, ring
 *            stages per warp, staged chunks per row, staged rows, segments one
 *            CTA may stage (decode kernel), grid, segment-list capacity, 1 if the
 *            prefill kernel runs it, dynamic shared memory bytes, and (if
 *            out_len >= 11) 1 if CTA ranges are aligned to K slices.
 * Returns NVFP4_ERR_SHAPE for shapes the product rejects or no plan fits.
 */
nvfp4_status nvfp4_plan_info(int32_t product, int32_t m, int32_t n, int32_t k, int32_t top_k, int32_t n_experts,
                             int32_t sms, int32_t *out, int32_t out_len);

/*
 * Host-side walk of the launch a product would make (same arguments as
 * nvfp4_plan_info) over n_seg segments, through the kernels' own work
 * decomposition code: every CTA, run, warp and piece.  No device work and no
 * CUDA call.
 *   out  (host) int32 [8]: 1 if every (segment, 64-row group, 16-row tile, K
 *        slice) is computed exactly once, every piece lies in its CTA's staged
 *        columns and segments (a prefill piece in its run's block), and every
 *        K-split counter in its fixed area (else 0); the largest staged column
 *        span; the planned span capacity; the most segments one CTA stages; the
 *        planned segment capacity; the tiles and the pieces walked; the dynamic
 *        shared memory bytes; and, if out_len >= 10, the most (16-row tile x
 *        64-column chunk) steps any warp of the decode kernel streams and the
 *        mean over all warps, rounded up (both 0 for the prefill kernel).
 * Returns NVFP4_ERR_SHAPE for rejected shapes or n_seg above the plan's capacity.
 */
nvfp4_status nvfp4_plan_check(int32_t product, int32_t m, int32_t n, int32_t k, int32_t top_k, int32_t n_experts,
                              int32_t sms, int32_t n_seg, int32_t *out, int32_t out_len);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_SKINNY_H_ */
