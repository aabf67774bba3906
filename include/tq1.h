/*
 * tq1.h -- C ABI of libtq1: ternary TQ1_0 weights x Q8_1 activations on
 * NVIDIA GB300 (sm_103a).
 *
 * Formats (PrismML-Eng/llama.cpp issue #139, "Current behavior": five trits
 * per byte in base 3, chunk c of a 256-element block reading digit c of
 * qs[0..31]; the block specification that accompanies it fixes the rest):
 *
 *   TQ1_0 block, 54 bytes, 256 weights:
 *     bytes  0..47  qs[48]  five trits per byte
 *     bytes 48..51  qh[4]   four trits per byte
 *     bytes 52..53  d       fp16 scale, little-endian
 *   byte b holding trits u0..u4 (u in {0,1,2}, u0 most significant) is
 *   ceil((sum u_i 3^(4-i)) * 256 / 243); digit k of b is ((uint8)(b*3^k)*3)>>8;
 *   trit 0/1/2 means weight -d/0/+d.  Element e of a block is
 *     e <  160: qs[e % 32] digit e / 32
 *     e <  240: qs[32 + (e - 160) % 16] digit (e - 160) / 16
 *     e >= 240: qh[(e - 240) % 4] digit (e - 240) / 4
 *   A matrix of n rows and k columns (k % 256 == 0) is [n][k/256] blocks,
 *   rows contiguous.
 *
 *   Q8_1 block, 36 bytes, 32 activations: fp16 d @0, fp16 s @2, int8 q[32] @4.
 *   A [t][k] activation matrix is [t][k/32] blocks.
 *
 *   TQ2_0 block, 66 bytes, 256 weights (the 2-bit sibling format the same
 *   page names in "Upstream state" without a layout; this library's reading):
 *     bytes  0..63  qs[64]  four 2-bit codes per byte, code = trit + 1
 *     bytes 64..65  d       fp16 scale, little-endian
 *   Element e of a block is field (e/32) % 4 (bits 2f..2f+1) of byte
 *   qs[32 * (e/128) + e % 32]: chunk c reads one field of 32 consecutive
 *   bytes, the chunk pattern above with four codes per byte.  Code 3 is never
 *   written and decodes to +2*d.
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller and must be
 *     16-byte aligned (TQ1_ERR_ALIGN otherwise).  The library never
 *     synchronises and allocates no device memory; work is enqueued on
 *     `stream` (a cudaStream_t, NULL for the legacy default stream) on the
 *     current device.  Scratch, where a path needs any, is a caller-owned
 *     workspace with a size query (tq1_mmv_ws, tq1_mmv_id).
 *   - Arguments are checked on the host before anything is launched; a
 *     failed check returns its negative code and launches nothing.
 *   - Shapes: k must be a positive multiple of 256; n, t >= 0 (0 means there
 *     is nothing to do and TQ1_OK is returned).
 *   - Errors met while kernels run (a bulk-copy wait that timed out, a
 *     routing id out of range) set a device status word; tq1_sync_status()
 *     synchronises `stream` and returns and clears it.
 *   - Kernels are launched with programmatic dependent launch: the mat-vec
 *     kernels start streaming weight blocks before the previous kernel in the
 *     stream has finished, so weight blocks must not be written by a kernel
 *     that lets its dependents start early (tq1_quantize_rows does not).
 */
#ifndef TQ1_H_
#define TQ1_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum tq1_status {
  TQ1_OK = 0,
  TQ1_ERR_NULL = -1,        /* a required pointer is NULL */
  TQ1_ERR_SHAPE = -2,       /* k not a positive multiple of 256, or n/t/top_k negative */
  TQ1_ERR_ALIGN = -3,       /* a pointer is not 16-byte aligned */
  TQ1_ERR_UNSUPPORTED = -4, /* shape beyond the kernels' limits (e.g. k > 62720) */
  TQ1_ERR_WORKSPACE = -5,   /* workspace too small */
  TQ1_ERR_CUDA = -6,        /* a CUDA runtime call failed */
  TQ1_ERR_TIMEOUT = -7,     /* a kernel gave up waiting on a transfer (device status) */
  TQ1_ERR_BAD_ID = -8       /* a routing id was outside [0, n_experts) (device status) */
};

/* Text for a status code (static storage).  No passage: a convention of this
 * library (the pages define no API). */
const char* tq1_status_string(int status);

/* Library version, e.g. "0.1.0".  No passage: a convention of this library. */
const char* tq1_version(void);

/*
 * Test hook for the error path of the bounded transfer waits.  The next
 * tq1_mmv / tq1_mmv_add / tq2_mmv / tq2_mmv_add call consumes the hook,
 * whichever kernel it runs; when that call runs the decode kernel
 * (1 <= t <= 5), its first CTA issues no copy (and no byte count) for its
 * first 4-row group, so every wait on that group gives up after about 2 s:
 * the call then reports TQ1_ERR_TIMEOUT through tq1_sync_status, its outputs
 * are unspecified, and the device and the library stay usable.  Nothing
 * faults, traps or hangs.  No passage: a convention of this library.
 */
void tq1_debug_inject_wait_timeout(void);

/* Name and text of the last CUDA runtime error this thread saw inside the
 * library (empty if none); explains a TQ1_ERR_CUDA.  No passage: a
 * convention of this library. */
const char* tq1_last_cuda_error(void);

/* Bytes of a TQ1_0 matrix [n][k/256], a TQ2_0 matrix [n][k/256] and a Q8_1
 * matrix [t][k/32] (54, 66 and 36 bytes per block, as the formats at the top
 * of this file lay them out).  No passage: a convention of this library. */
size_t tq1_blocks_bytes(int64_t n, int64_t k);
size_t tq2_blocks_bytes(int64_t n, int64_t k);
size_t tq1_q8_1_bytes(int64_t t, int64_t k);

/*
 * Quantise fp32 weights w[n][k] (row-major) to TQ1_0 blocks.
 * Per 256-weight block: d = fp16(max |w|); trit = clamp(round_half_away(w / max|w|),
 * -1, 1), or 0 when the block is all zero.  Bit-exact, deterministic.
 * Source: PrismML-Eng/llama.cpp issue #139, "Current behavior" (the block
 * format); the rounding is this library's reading (the pages do not state
 * one).
 */
int tq1_quantize_rows(const float* w, void* blocks, int64_t n, int64_t k, void* stream);

/*
 * Quantise fp32 activations x[t][k] to Q8_1 blocks q8[t][k/32].
 * Per 32-value block: d = max|x| / 127 (fp32); q = clamp(round_half_away(x / d),
 * -127, 127), or 0 when d == 0; stored fp16(d), fp16(d * sum q), q.
 * k must be a positive multiple of 32 here.  Bit-exact, deterministic.
 * Source: PrismML-Eng/llama.cpp issue #139, "Current behavior" (the Q8_1
 * activation blocks of 32 values whose per-block dot product the mat-vec
 * computes); the rounding is this library's reading (the pages do not state
 * one).
 */
int q8_1_quantize_acts(const float* x, void* q8, int64_t t, int64_t k, void* stream);

/*
 * Mat-vec for t token columns: y[c][r] = sum_k w[r][k] * x[c][k] with
 * w = d_w * trit and x = d_a * q, accumulated as
 *   sum_blocks d_w * sum_{chunks j} d_a[j] * I_j,   I_j = sum (trit * q) (exact int32)
 * in fp32.  blocks [n][k/256] TQ1_0, q8 [t][k/32] Q8_1, y fp32 [t][n].
 * The ladder: t <= 5 runs the byte-major dp4a decode kernel (rungs of
 * 1/2/4/8 columns); t >= 6 runs the warp-level tensor-core kernel (mma.sync
 * on exact fp16 operands, trit-derived and the int8 q, with an fp32
 * accumulation of each 32-element chunk that is exact) with rungs of
 * 8/16/24/32 token columns,
 * in slices of 32 columns above 32; shapes either cannot stage take a
 * general dp4a kernel.  Nothing
 * is allocated; for prefill-sized t, tq1_mmv_ws with a workspace runs the
 * tcgen05 tile path instead.  Deterministic: repeated calls give identical
 * bits.
 * Source: PrismML-Eng/llama.cpp issue #139, "Proposed approach" (a dedicated
 * whole-block kernel that iterates over packed bytes); laddered column
 * counts: Neroued/ninfer issue #293.
 */
int tq1_mmv(const void* blocks, const void* q8, float* y, int64_t n, int64_t k, int64_t t, void* stream);

/*
 * Workspace bytes tq1_mmv_ws / tq2_mmv_ws need for an n x k matrix and t
 * columns: the tcgen05 tile path's exact fp16 hi/lo split of the activations
 * (2 * 2 * t_pad * k + 4 * t_pad bytes, t_pad = t rounded up to the token
 * tile, rounded up to 256).  0 when the call takes the allocation-free
 * kernels (t below the tile path's threshold, or a row stride that is not a
 * multiple of 16 bytes, i.e. k not a multiple of 2048).
 * Source: PrismML-Eng/llama.cpp issue #139, "Measured impact" (prefill, pp512,
 * is the case the dense tensor-core path serves); the workspace itself is a
 * convention of this library.
 */
size_t tq1_mmv_workspace_size(int64_t n, int64_t k, int64_t t);

/*
 * tq1_mmv / tq1_mmv_add with a caller-owned workspace: where
 * tq1_mmv_workspace_size(n, k, t) > 0 (prefill-sized t), a prep kernel
 * splits the activations into exact fp16 hi/lo rows in `ws` and a tcgen05
 * kernel (A: the weights expanded straight into tensor memory; B: the hi/lo
 * rows by TMA; fp32 accumulators in tensor memory) contracts them; otherwise
 * the call equals tq1_mmv (res == NULL) or tq1_mmv_add.  res may be NULL or
 * y itself.  ws: device, 16-byte aligned, at least
 * tq1_mmv_workspace_size(n, k, t) bytes (TQ1_ERR_WORKSPACE otherwise; checked
 * before any launch), or NULL (then the allocation-free kernels run).  The
 * workspace is in use until the call's kernels finish on `stream`.
 * tq2_mmv_ws: the same for TQ2_0 weights.
 * Source: PrismML-Eng/llama.cpp issue #139, "Measured impact" and
 * "Proposed approach" (prefill through a dedicated whole-block kernel).
 */
int tq1_mmv_ws(const void* blocks, const void* q8, const float* res, float* y, int64_t n, int64_t k, int64_t t,
               void* ws, size_t ws_bytes, void* stream);
int tq2_mmv_ws(const void* blocks, const void* q8, const float* res, float* y, int64_t n, int64_t k, int64_t t,
               void* ws, size_t ws_bytes, void* stream);

/*
 * Decode mat-vec straight from fp32 activations: the Q8_1 quantisation of x
 * (the same operations and rounding as q8_1_quantize_acts) runs in the dp4a
 * decode kernel's prologue, so a decode step needs one launch per mat-vec
 * instead of two.  y equals, bit for bit, q8_1_quantize_acts followed by
 * tq1_mmv (the same decode kernel on the same records).  x: fp32 [t][k],
 * device, 16-byte aligned.  1 <= t <= 4 (larger t: TQ1_ERR_UNSUPPORTED; quantise
 * once and call tq1_mmv).  Errors as tq1_mmv.
 * Source: PrismML-Eng/llama.cpp issue #139, "Current behavior" (activations
 * are quantised to Q8_1 before the MMVQ kernel: here inside it).
 */
int tq1_mmv_f32(const void* blocks, const float* x, float* y, int64_t n, int64_t k, int64_t t, void* stream);

/*
 * Mat-vec with a residual added in the kernel's epilogue:
 *   y[c][r] = res[c][r] + sum_k w[r][k] * x[c][k]
 * (one fp32 add per output after the dot product; the same kernels, rungs and
 * accumulation as tq1_mmv).  res: fp32 [t][n], device, 16-byte aligned; it may
 * be y itself (in-place update).  Errors as tq1_mmv; res == NULL is
 * TQ1_ERR_NULL.
 * Source: Neroued/ninfer issue #293 (the linear_add rungs: a linear layer
 * fused with its residual add).
 */
int tq1_mmv_add(const void* blocks, const void* q8, const float* res, float* y, int64_t n, int64_t k, int64_t t,
                void* stream);

/*
 * Debug entry: the exact integer partials part[c][r][j] = I_j (int32,
 * [t][n][k/32]) that tq1_mmv scales, for any t, from the kernel tq1_mmv runs
 * for that t: the dp4a decode kernel at t <= 5 (its dp4a sums, stored before
 * scaling), the tensor-core rungs at t >= 6 (each chunk's accumulator, which
 * holds exactly I_j when the operands are unscaled); shapes neither can stage
 * take the general kernel.  Bit-exact by construction.
 * Source: PrismML-Eng/llama.cpp issue #139, "Acceptance criteria" (the new
 * kernel checked case by case against a CPU reference), and the per-32-block
 * integer dot product of "Current behavior" that the kernels compute.
 */
int tq1_mmv_partials(const void* blocks, const void* q8, int32_t* part, int64_t n, int64_t k, int64_t t,
                     void* stream);

/*
 * Dequantise TQ1_0 rows: out[r][j] = d_w(r, j/256) * trit(r, j), the value the
 * block encodes (fp32 when out_f16 == 0, else fp16; both exact, since the
 * scale is an fp16 value and the trit is -1, 0 or +1).
 *   blocks: [n][k/256] TQ1_0;  out: [n][k] fp32 or fp16, 16-byte aligned.
 * Source: PrismML-Eng/llama.cpp issue #139, "Current behavior" (the CPU
 * dequantize_row walk: each packed byte amortised over its trits, element
 * order of the block) and "Upstream state" (the dequant shader that ships with
 * the Vulkan mat-vec).
 */
int tq1_dequantize_rows(const void* blocks, void* out, int64_t n, int64_t k, int out_f16, void* stream);

/*
 * Gather dequantised rows (get_rows, e.g. an embedding lookup):
 * out[i][:] = row row_ids[i] of the n x k TQ1_0 matrix, i < n_ids, fp32 or
 * fp16 as in tq1_dequantize_rows.  An id outside [0, n) leaves its output row
 * untouched and sets TQ1_ERR_BAD_ID in the device status (tq1_sync_status).
 *   row_ids: int32 [n_ids] (device);  out: [n_ids][k].
 * Source: PrismML-Eng/llama.cpp issue #139, "Upstream state" (get_rows for the
 * format next to its mat-vec).
 */
int tq1_get_rows(const void* blocks, const int32_t* row_ids, int64_t n_ids, void* out, int64_t n, int64_t k,
                 int out_f16, void* stream);

/*
 * Workspace bytes tq1_mmv_id needs for n_experts experts and t*top_k routed
 * pairs (the compacted routing table: n_active, expert bounds, active
 * experts, sorted pairs, task offsets).  Small routings (four words per
 * expert plus one per pair within 16 KiB) build the table inside the routed
 * kernel and leave the workspace untouched; it is required all the same.
 * Source: AMD-Ecosystem/llama.cpp PR #76, "Summary" (ids -> expert_bounds ->
 * compacted grid: the table this workspace holds).
 */
size_t tq1_mmv_id_workspace_size(int64_t n_experts, int64_t t, int64_t top_k);

/*
 * Expert-routed mat-vec (MoE "mul_mat_id"): y[c][s][r] = expert ids[c][s]'s
 * matrix times token c's activations, for every token c < t and slot s < top_k.
 *   expert_blocks: n_experts matrices [n][k/256] back to back (expert e starts
 *                  at byte e * tq1_blocks_bytes(n, k))
 *   q8:            [t][k/32] Q8_1, one row per token (shared by its slots)
 *   ids:           int32 [t][top_k] expert ids
 *   y:             fp32 [t][top_k][n]
 *   ws, ws_bytes:  caller-owned device workspace of at least
 *                  tq1_mmv_id_workspace_size() bytes (TQ1_ERR_WORKSPACE otherwise);
 *                  it holds the compacted routing table between the two launches.
 * Ids outside [0, n_experts) skip their slot (its output is left untouched) and
 * set TQ1_ERR_BAD_ID in the device status.  n_experts <= 12288.
 * Source: AMD-Ecosystem/llama.cpp PR #76, "Summary" (ids -> expert_bounds ->
 * compacted grid); PrismML-Eng/llama.cpp issue #139, "Acceptance criteria"
 * (MUL_MAT_ID with fewer experts used than available).
 */
int tq1_mmv_id(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids, float* y,
               int64_t n, int64_t k, int64_t t, int64_t top_k, void* ws, size_t ws_bytes, void* stream);

/*
 * Expert-routed mat-vec with one activation row per routed (token, slot) pair
 * (the down-projection of an expert layer, whose input differs per slot):
 *   y[c][s][r] = expert ids[c][s]'s matrix times activation row (c, s).
 *   q8: [t][top_k][k/32] Q8_1.  Everything else, including the workspace and
 * the error behaviour, as tq1_mmv_id.
 * Source: PrismML-Eng/llama.cpp issue #139, "Acceptance criteria" (MUL_MAT_ID
 * cases); AMD-Ecosystem/llama.cpp PR #76, "Summary" (ids -> expert bounds ->
 * compacted grid).
 */
int tq1_mmv_id_slots(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids, float* y,
                     int64_t n, int64_t k, int64_t t, int64_t top_k, void* ws, size_t ws_bytes, void* stream);

/*
 * Debug entry: the exact integer partials part[c][s][r][j] = I_j (int32,
 * [t][top_k][n][k/32]) that tq1_mmv_id / tq2_mmv_id scale, from the routed
 * decode kernels themselves (their expansion and dp4a sums, stored before
 * scaling): direct mode for up to 128 routed pairs, the compacted mode above.
 * Arguments, workspace and errors as tq1_mmv_id (part replaces y); shapes
 * that only the general kernel can stage return TQ1_ERR_UNSUPPORTED.
 * Source: AMD-Ecosystem/llama.cpp PR #76, "Summary" (the expert-routed grid
 * these kernels run); PrismML-Eng/llama.cpp issue #139, "Acceptance criteria"
 * (MUL_MAT_ID checked against a CPU reference).
 */
int tq1_mmv_id_partials(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids,
                        int32_t* part, int64_t n, int64_t k, int64_t t, int64_t top_k, void* ws, size_t ws_bytes,
                        void* stream);
int tq2_mmv_id_partials(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids,
                        int32_t* part, int64_t n, int64_t k, int64_t t, int64_t top_k, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * tq1_mmv_id without a workspace argument, for callers that cannot allocate
 * device memory (inside a stream capture, under a fixed memory budget, in a
 * latency-critical loop, or from plain C with no allocator at hand).  The
 * routing table lives in a fixed array that is part of the library image
 * (about 76 KiB on every GPU that loads the library, held until exit).
 * Limits: n_experts <= 1024 and t * top_k <= 16384; larger calls return
 * TQ1_ERR_WORKSPACE and launch nothing.  Same arguments, layouts, results
 * and errors as tq1_mmv_id otherwise.
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture begins.
 * All calls on a device share the array (each call rewrites what it reads,
 * so nothing needs clearing); calls that may overlap on the GPU race on it.
 * No passage: a convention of this library (the pages have no counterpart
 * to this entry point).
 */
int tq1_mmv_id_noalloc(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids, float* y,
                       int64_t n, int64_t k, int64_t t, int64_t top_k, void* stream);

/*
 * Synchronise `stream`, then return and clear the device status word:
 * TQ1_OK, TQ1_ERR_TIMEOUT or TQ1_ERR_BAD_ID (or TQ1_ERR_CUDA if the stream
 * itself reported an error).  No passage: a convention of this library (the
 * pages define no error reporting).
 */
int tq1_sync_status(void* stream);

/*
 * TQ2_0 weights (2-bit codes; format at the top of this file).
 *
 * tq2_quantize_rows: fp32 w[n][k] -> TQ2_0 blocks, with the same scale and
 * trit rounding as tq1_quantize_rows (so both formats hold the same trits and
 * scales for the same weights).  Bit-exact, deterministic.
 *
 * tq2_mmv: y[c][r] = sum_k w[r][k] * x[c][k] for TQ2_0 blocks [n][k/256] and
 * Q8_1 q8 [t][k/32], accumulated exactly as tq1_mmv (exact int32 per-32
 * partials, fp32 scale-and-sum per block).  The same ladder as tq1_mmv:
 * t <= 5 runs the decode kernel (the codes already are its packed-digit
 * registers: masked dp4a, no expansion), t >= 6 the warp-level tensor-core
 * rungs (the codes become fp16 operands by a byte permute), with the
 * tcgen05 tile path through tq2_mmv_ws.  Deterministic; allocates nothing.
 *
 * tq2_mmv_partials: the exact int32 partials part[c][r][k/32] of tq2_mmv
 * (debug, as tq1_mmv_partials).
 *
 * Arguments, alignment, shapes and errors as the TQ1_0 counterparts.
 * Source: PrismML-Eng/llama.cpp issue #139, "Upstream state" (TQ2_0 as the
 * stalled sibling of the TQ1_0 port) and "Proposed approach" (whole-block
 * kernels that load each packed byte once).
 */
int tq2_quantize_rows(const float* w, void* blocks, int64_t n, int64_t k, void* stream);
int tq2_mmv(const void* blocks, const void* q8, float* y, int64_t n, int64_t k, int64_t t, void* stream);
int tq2_mmv_partials(const void* blocks, const void* q8, int32_t* part, int64_t n, int64_t k, int64_t t,
                     void* stream);

/*
 * TQ2_0 counterparts of tq1_mmv_f32 (Q8_1 quantisation fused into the decode
 * kernel's prologue, 1 <= t <= 4, bit-identical to q8_1_quantize_acts +
 * tq2_mmv) and tq1_mmv_add (y = res + W x, res may be y).  Arguments and
 * errors as those.
 * Source: as tq1_mmv_f32 and tq1_mmv_add, with PrismML-Eng/llama.cpp issue
 * #139, "Upstream state" (the TQ2_0 sibling format).
 */
int tq2_mmv_f32(const void* blocks, const float* x, float* y, int64_t n, int64_t k, int64_t t, void* stream);
int tq2_mmv_add(const void* blocks, const void* q8, const float* res, float* y, int64_t n, int64_t k, int64_t t,
                void* stream);

/*
 * TQ2_0 rows to fp32 (out_f16 == 0) or fp16 values, d * (code - 1) exactly:
 * the whole matrix (tq2_dequantize_rows) or the rows listed in row_ids
 * (tq2_get_rows).  Arguments, layouts, errors and the handling of
 * out-of-range ids as tq1_dequantize_rows / tq1_get_rows.
 * Source: PrismML-Eng/llama.cpp issue #139, "Upstream state" (the TQ2_0
 * sibling format) and "Current behavior" (the dequantise walk of a block).
 */
int tq2_dequantize_rows(const void* blocks, void* out, int64_t n, int64_t k, int out_f16, void* stream);
int tq2_get_rows(const void* blocks, const int32_t* row_ids, int64_t n_ids, void* out, int64_t n, int64_t k,
                 int out_f16, void* stream);

/*
 * Expert-routed mat-vec over TQ2_0 experts (each expert [n][k/256] x 66
 * bytes, back to back): the same routing, workspace
 * (tq1_mmv_id_workspace_size), kernels, layouts and errors as tq1_mmv_id
 * (one activation row per token) and tq1_mmv_id_slots (one per token and
 * slot).
 * Source: AMD-Ecosystem/llama.cpp PR #76, "Summary" (ids -> expert_bounds ->
 * compacted grid); PrismML-Eng/llama.cpp issue #139, "Upstream state" (the
 * TQ2_0 sibling format).
 */
int tq2_mmv_id(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids, float* y,
               int64_t n, int64_t k, int64_t t, int64_t top_k, void* ws, size_t ws_bytes, void* stream);
int tq2_mmv_id_slots(const void* expert_blocks, int64_t n_experts, const void* q8, const int32_t* ids, float* y,
                     int64_t n, int64_t k, int64_t t, int64_t top_k, void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ1_H_ */
