/*
 * gq.h -- C ABI of libgq: block-quantized matrix-vector products for GB300
 * (sm_103a) with the dequantization fused in, their epilogues, and the
 * Q4_0 x Q8_0 prefill contraction.
 *
 * Sources (page title, section):
 *   "Gemma 4 M4 Max kernel roadmap" (gem, docs/research/kernel-roadmap.md),
 *       K2 "Metal decode path": the decode steps in order -- a Q4_0
 *       matrix-vector product with fused dequantization and F32
 *       accumulation (step 1), the gated GELU FFN projection pair (step 5),
 *       the Q8_0 embedding/output projection with on-GPU top-k (step 6);
 *       K3 "prefill path": batched Q4_0 matrix-matrix kernels;
 *       K4 "scheduling and memory": arenas are allocated once and
 *       generation performs no tensor-sized allocation.
 *   "Metal kernel capability table (Phase B ground truth)", section 1
 *       "Quant matvec family" (Q4_0 18 B, Q4_K 144 B, Q8_0 blocks; legal K
 *       and tail handling), section 9 (legal dimensions are checked at
 *       dispatch, not assumed; one explicit kernel per format), section 8
 *       findings F4, F6 and F17 (silent no-ops and silent truncation are
 *       defects).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are caller-owned DEVICE memory, 16-byte aligned
 *     (packed Q8_0 weights: 32-byte aligned, for 32-byte loads).
 *     The library allocates nothing, never synchronizes the device, and
 *     launches only on `stream` (NULL = the legacy default stream).
 *   - Argument errors are reported before any launch as a negative gq_status;
 *     nothing is launched and no output is touched.  After a launch,
 *     a CUDA launch error is returned as GQ_ERR_CUDA.
 *   - rows, K, M are element counts.  K must be whole blocks (a multiple of
 *     32; of 256 for Q4_K); K is never silently truncated.  Rows need not
 *     divide any tile: the row tail is masked inside the kernels.
 *   - Weights W are in the PACKED layout written by gq_pack (same byte count
 *     as the canonical GGUF-order blocks; see gq_pack).
 *   - Results are deterministic: the same inputs give bitwise the same
 *     outputs on the same GPU and launch configuration.
 *   - The decode kernels may start while the preceding kernel in `stream`
 *     is still running (programmatic dependent launch).  They read their
 *     activation inputs and write their outputs only after that kernel has
 *     completed, but they may read the packed weights W earlier: weights
 *     are constants of the model.  W must therefore not be written by the
 *     kernel that immediately precedes the call in `stream`, unless that
 *     kernel is gq_pack's (which makes its writes visible before it exits).
 */
#ifndef GQ_H
#define GQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* identical to cudaStream_t */
typedef struct CUstream_st *gq_stream_t;

typedef enum {
    GQ_OK = 0,
    GQ_ERR_NULL = -1,      /* a required pointer is NULL */
    GQ_ERR_ALIGN = -2,     /* a pointer is not 16-byte aligned */
    GQ_ERR_SHAPE = -3,     /* rows/K/M/k outside the legal range */
    GQ_ERR_WORKSPACE = -4, /* workspace missing or too small */
    GQ_ERR_CUDA = -5,      /* the CUDA runtime reported an error */
    GQ_ERR_TIMEOUT = -6,   /* a bounded in-kernel wait gave up */
    GQ_ERR_FORMAT = -7     /* unknown block format */
} gq_status;

enum {
    GQ_FORMAT_Q4_0 = 0, /* 18 B / 32 weights: fp16 d, 16 B nibbles; w = (q - 8) d   */
    GQ_FORMAT_Q8_0 = 1, /* 34 B / 32 weights: fp16 d, 32 int8 q;     w = q d        */
    GQ_FORMAT_Q4_K = 2, /* 144 B / 256 weights: fp16 d, dmin, 12 B 6-bit sc/m,
                           128 B nibbles;                       w = d sc q - dmin m */
    GQ_FORMAT_Q6_K = 3  /* 210 B / 256 weights: 128 B low 4 code bits, 64 B top 2
                           bits, 16 int8 sub-scales, fp16 d; w = d sc (q - 32) */
};

/* Largest K accepted by the single-pass matvec kernels (the whole activation
 * vector is staged in shared memory). */
#define GQ_MAX_K 49152
/* Largest k accepted by gq_logits_topk. */
#define GQ_MAX_TOPK 64

/* Human-readable name of a gq_status value (static storage). */
const char *gq_status_string(int status);

/* ---------------------------------------------------------------------------
 * Packing (one-time, not on the decode path).
 *
 * The canonical blocks are the GGUF byte order: Q4_0 byte j holds element j
 * (low nibble) and element j+16 (high nibble); Q4_K's 128 nibble bytes are
 * four 32-byte chunks, chunk c holding sub-block 2c in the low nibbles and
 * 2c+1 in the high nibbles; Q6_K's code bits follow the GGUF placement (in
 * each 128-weight half, weight 32c + l has its low 4 bits in ql byte
 * l + 32(c % 2) of the half, low nibble for c < 2, and its top 2 bits at bit
 * 2c of qh byte l of the half).  The packed layout keeps every bit of every
 * block and the same total byte count; it is a bijection, undone exactly by
 * gq_unpack.  Packed layout of a rows x K matrix with nb blocks per row:
 *   Q4_0: plane 0 = rows*nb 16-byte payloads, row-major, nibbles in element
 *         order (byte i = element 2i low, 2i+1 high); plane 1 = rows*nb fp16
 *         scales d, row-major.
 *   Q8_0: plane 0 = rows*nb 32-byte payloads, each byte q XOR 0x80
 *         (offset binary); plane 1 = rows*nb fp16 scales d.
 *   Q4_K: plane 0 = rows*ns 128-byte payloads (ns super-blocks per row),
 *         sub-block s at bytes 16s..16s+15, nibbles in element order;
 *         plane 1 = rows*ns 16-byte records {d, dmin, 12 scale bytes}
 *         copied unchanged.
 *   Q6_K: plane 0 = rows*ns 128-byte low-bit payloads in element order;
 *         plane 1 = rows*ns 64-byte top-bit payloads of 16 little-endian
 *         32-bit words, word g holding elements 16g..16g+15: element
 *         16g + 4a + i (a, i = 0..3) at bits p, p+1 with
 *         p = 4i + {0, 2, 16, 18}[a]; plane 2 = rows*ns 16-byte int8
 *         sub-scale records; plane 3 = rows*ns fp16 d (both copied
 *         unchanged).
 * W_canon and W_packed must not overlap.  Both are device pointers.
 * ------------------------------------------------------------------------ */
size_t gq_packed_bytes(int format, int rows, int K); /* 0 if invalid */
int gq_pack(int format, const void *W_canon, void *W_packed, int rows, int K,
            gq_stream_t stream);
int gq_unpack(int format, const void *W_packed, void *W_canon, int rows, int K,
              gq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Decode matvecs: y[i] = sum_j w_ij x_j with w decoded from the block and all
 * arithmetic in f32 ("Gemma 4 M4 Max kernel roadmap", K2 step 1; "Metal
 * kernel capability table", section 1, q4_f32_matvec / q4k_matvec rows).
 *   W  packed weights, rows x K   x  f32[K]   y  f32[rows] (overwritten)
 *   M  batch size; must be 1 (decode).  1 <= rows, 32 <= K <= GQ_MAX_K.
 * Accuracy: |y_i - exact_i| <= 1e-5 * sum_j |w_ij x_j| for finite inputs.
 * gq_q4k_matvec works in a domain scaled by a power of two taken from the
 * largest finite |x_j| = X: the bound holds for elements with
 * |x_j| >= 2^-104 * X; a product involving a smaller element is rounded to
 * an absolute grid of at most 2^-128 * X * |d * sc|.  Scaling x by 2^k scales
 * y by exactly 2^k while nothing over- or underflows.
 * Non-finite x: y_i is non-finite exactly where the definition's sum is.
 * Q4_0, Q8_0 and Q6_K also give the definition's NaN or infinity; Q4_K forms
 * each sub-block as d*sc*sum(q x) - dmin*m*sum(x), so an infinity that meets
 * a zero code or the min term can give NaN where the per-weight sum is
 * infinite.
 * ------------------------------------------------------------------------ */
int gq_q4_0_matvec(const void *W, const float *x, float *y, int rows, int K, int M,
                   gq_stream_t stream);
int gq_q8_0_matvec(const void *W, const float *x, float *y, int rows, int K, int M,
                   gq_stream_t stream);
int gq_q4k_matvec(const void *W, const float *x, float *y, int rows, int K, int M,
                  gq_stream_t stream);
/* Q6_K ("Metal kernel capability table", section 1, q6k_matvec row: 210-byte
 * super-blocks, K % 256): w = d * sc[j / 16] * (q_j - 32) within a
 * super-block.  Same contract as the other matvecs. */
int gq_q6k_matvec(const void *W, const float *x, float *y, int rows, int K, int M,
                  gq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Gated GELU FFN gate/up pair ("Gemma 4 M4 Max kernel roadmap", K2 step 5;
 * "Metal kernel capability table", section 4 FFN family):
 *   g = W_gate x, u = W_up x (both Q4_0, rows x K, packed), and
 *   h[i] = gelu_tanh(g[i]) * u[i],
 *   gelu_tanh(a) = 0.5 a (1 + tanh(sqrt(2/pi) (a + 0.044715 a^3))), the tanh
 *   argument clamped to +-15 (finite for every finite a).
 * One pass over x, two weight streams.  h is f32[rows].  M must be 1.
 * The down projection is gq_q4_0_matvec with x = h.
 * ------------------------------------------------------------------------ */
int gq_ffn_gate_up_gelu(const void *W_gate, const void *W_up, const float *x, float *h,
                        int rows, int K, int M, gq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Tied-embedding Q8_0 logits with soft-cap and on-GPU top-k
 * ("Gemma 4 M4 Max kernel roadmap", K2 step 6; K1 logit soft-capping;
 * K5 device top-k with (value, token) pair frontiers):
 *   l[i] = sum_j w_ij x_j (W: Q8_0, rows x K, packed),
 *   l'[i] = softcap * tanh(l[i] / softcap)   (softcap <= 0: l' = l),
 *   idx[0..k), val[0..k) = the k largest l' in descending order; equal
 *   values rank by the lower row index; NaN ranks below every number;
 *   -0 ranks equal to +0.
 *   logits_or_null: if not NULL, receives l' for every row (f32[rows]).
 *   workspace: device scratch of at least gq_logits_topk_workspace_bytes
 *   bytes (caller-owned).  ZERO-FILL IT ONCE before its first use: its first
 *   16 bytes count the CTAs that have finished (the last one merges every
 *   CTA's candidates), and every completed call leaves that count at zero
 *   again, so the workspace can be reused without clearing.  The rest needs
 *   no initialisation.  Two calls that may run concurrently must not share
 *   it.
 *   1 <= k <= min(GQ_MAX_TOPK, rows); M must be 1.
 * One kernel is launched on `stream`.
 * ------------------------------------------------------------------------ */
size_t gq_logits_topk_workspace_bytes(int rows, int K, int k);
int gq_logits_topk(const void *W, const float *x, float softcap, int k, int *idx, float *val,
                   float *logits_or_null, void *workspace, size_t workspace_bytes, int rows,
                   int K, int M, gq_stream_t stream);

/* The same computation without the workspace argument, for callers that
 * cannot allocate device memory (a serving loop that must not call cudaMalloc
 * while it runs, a runtime that hands the library only its inputs and
 * outputs).  The source pages have no counterpart of this entry point.  The
 * per-CTA key lists live in a fixed 1 MiB array inside libgq (zero at load,
 * so it needs no clearing; held on every
 * GPU that loads the library until the process exits); every call
 * gq_logits_topk accepts fits, and a call that would not fit is rejected with
 * GQ_ERR_SHAPE.  The first call on a device looks the array's address up
 * (cudaGetSymbolAddress) -- make that first call before any stream capture.
 * The address is kept for the life of the process: do not call this entry
 * point again after cudaDeviceReset (or any other re-creation of the
 * device's primary context), which would leave it stale.
 * Calls share the array: calls that may overlap on the GPU race on it.
 * Nothing is allocated. */
int gq_logits_topk_noalloc(const void *W, const float *x, float softcap, int k, int *idx, float *val,
                           float *logits_or_null, int rows, int K, int M, gq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Q8_0 activation quantization ("Metal kernel capability table", section 2,
 * quantize_q8: f32 -> int8 plus per-32 scales; finding F6):
 *   for every token t < M and 32-block b of X[t, 0..K):
 *     amax = max |x|, d = amax / 127 (IEEE f32 division),
 *     q = clamp(round_half_away(x / d), -127, 127), and q = 0 when d = 0.
 *   X f32[M][K] row-major, Xq int8[M][K], dx f32[M][K/32].  Bit-exact.
 * ------------------------------------------------------------------------ */
int gq_quantize_q8_0(const float *X, int8_t *Xq, float *dx, int K, int M, gq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Prefill contraction ("Gemma 4 M4 Max kernel roadmap", K3 batched Q4_0
 * matrix-matrix) of packed Q4_0 weights W (rows x K) with Q8_0 activations
 * (Xq int8[M][K], dx f32[M][K/32], as written by gq_quantize_q8_0):
 *   D[t][r][b] = sum_{j<32} Xq[t][32b+j] * (q_w[r][32b+j] - 8)   (exact integers)
 *   Y[t][r]    = sum_b d_w[r][b] * dx[t][b] * D[t][r][b]          (f32)
 * Y is f32[M][rows] row-major (one row of Y per token).
 *
 * Y is computed on the tensor cores in one of three ways, all equal to the
 * sum above up to f32 rounding (|Y - Y_ref| <= 1e-5 * sum_k |w x| over the
 * dequantized operands w = d_w*(q_w-8), x = dx*Xq):
 *   K % 256 == 0, M <= 112: each block's exact integer D is formed by
 *     mma.sync on f16 operands holding the small integers and folded at once
 *     as Y += (d_w*dx)*D in f32, block by block (this also meets the tighter
 *     |Y - Y_ref| <= 1e-5 * sum_b |d_w dx D|);
 *   K % 256 == 0, M > 112: both block scales are folded, per 8-block chunk
 *     and with power-of-two chunk factors, into f16 operand pieces (dx*Xq as
 *     two, d_w*(q_w-8) as two exact pieces) and Y accumulates a chunk at a
 *     time in tensor memory (with more than 128 tokens on pairs of SMs);
 *   other K: each block's exact integer D is read out of tensor memory and
 *     folded in f32 (up to 24 tokens: the same D by dp4a on the CUDA cores).
 * Non-finite scales (dx from a non-finite X, or an fp16 d_w that is infinite
 * or NaN): Y[t][r] is non-finite exactly where the definition's sum is; the
 * exact-D paths give the definition's NaN or infinity, the scale-folded path
 * gives NaN for every such output (its pieces' difference of infinities).
 *
 * The workspace (device memory, 16-byte aligned, at least
 * gq_q4_0_gemm_workspace_bytes(K, M) bytes, owned by the caller) receives
 * the activation operands converted once for the tensor cores; its
 * contents are scratch before and after the call.  Two calls in flight at
 * the same time need two workspaces.  GQ_ERR_WORKSPACE if it is too small.
 * ------------------------------------------------------------------------ */
size_t gq_q4_0_gemm_workspace_bytes(int K, int M); /* 0 if K or M is invalid */
int gq_q4_0_gemm_q8act(const void *W, const int8_t *Xq, const float *dx, float *Y, void *workspace,
                       size_t workspace_bytes, int rows, int K, int M, gq_stream_t stream);

/* The integer block dot products of the same contraction, as the tensor-core
 * path computes them: D int32[M][rows][K/32] (D[t][r][b] above), exact.
 * Meant for checking small problems (the output is M*rows*K/32 words).
 * Same workspace rule as gq_q4_0_gemm_q8act. */
int gq_q4_0_gemm_block_dots(const void *W, const int8_t *Xq, int32_t *D, void *workspace,
                            size_t workspace_bytes, int rows, int K, int M, gq_stream_t stream);

/* ---------------------------------------------------------------------------
 * Device status: GQ_ERR_TIMEOUT if a kernel launched since the last reset
 * gave up one of its bounded in-kernel waits (its outputs are then invalid),
 * else GQ_OK; GQ_ERR_CUDA if the status cannot be read.  This call
 * SYNCHRONIZES with the device.  reset != 0 clears the status.
 * ------------------------------------------------------------------------ */
int gq_device_status(int reset);

/* Self-check of the bounded-wait path of the tensor-core kernels: launches
 * one CTA whose thread waits, with the kernels' wait helper and time limit
 * (about 2 s), on an mbarrier phase that nothing completes.  The wait gives
 * up, records GQ_ERR_TIMEOUT in the device status (read it with
 * gq_device_status) and the kernel returns normally; the context stays
 * usable.  Returns the launch status.  For tests. */
int gq_selftest_bounded_wait(gq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GQ_H */
