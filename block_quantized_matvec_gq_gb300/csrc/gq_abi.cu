// gq_abi.cu -- the exported C entry points: argument validation, then launch.
//
// "Metal kernel capability table (Phase B ground truth)", section 9: legal
// dimensions are checked at dispatch, not assumed; section 8, findings F4,
// F6, F17: a silent no-op or a silently truncated K is a defect.  Every
// entry point here rejects what its kernels cannot compute exactly, before
// launching anything.
#include <math.h>

#include "gq_geglu.h"
#include "gq_host.h"
#include "gq_norm.h"

using namespace gq;

// Launchers of the entry points declared in gq_geglu.h and gq_norm.h.  They
// are declared here rather than in gq_host.h, which every kernel includes,
// so that adding them changed no other kernel's sources (whose recorded DRAM
// counters are keyed to a digest of those sources).
namespace gq {
// gq_q4_0.cu: the Q4_0 matvec staging gelu_tanh(g) * u as its input vector
int launch_q4_0_geglu_down(const void *W, const float *g, const float *u, float *y, int rows, int K, MatvecGeo geo,
                           cudaStream_t s);
// gq_norm.cu: RMS normalization fused with Q8_0 quantization, one CTA per token
int launch_rmsnorm_q8_0(const float *X, const float *w, float offset, float eps, int8_t *Xq, float *dx, int K,
                        int M, cudaStream_t s);
// gq_norm.cu: the exact sum of squares of every row
int launch_row_sum_squares(const float *X, double *ss, int K, int M, cudaStream_t s);
}  // namespace gq

namespace {

int block_weights(int format) { return (format == GQ_FORMAT_Q4_K || format == GQ_FORMAT_Q6_K) ? 256 : 32; }

int block_bytes(int format)
{
    switch (format) {
    case GQ_FORMAT_Q4_0: return 18;
    case GQ_FORMAT_Q8_0: return 34;
    case GQ_FORMAT_Q4_K: return 144;
    case GQ_FORMAT_Q6_K: return 210;
    }
    return 0;
}

bool valid_format(int format)
{
    return format == GQ_FORMAT_Q4_0 || format == GQ_FORMAT_Q8_0 || format == GQ_FORMAT_Q4_K ||
           format == GQ_FORMAT_Q6_K;
}

int check_matvec(int format, const void *W, const float *x, const float *y, int rows, int K, int M)
{
    if (!W || !x || !y) return GQ_ERR_NULL;
    if (!aligned16(W) || !aligned16(x) || !aligned16(y)) return GQ_ERR_ALIGN;
    if (rows < 1 || M != 1 || K < block_weights(format) || K % block_weights(format) != 0 || K > GQ_MAX_K)
        return GQ_ERR_SHAPE;
    return GQ_OK;
}

}  // namespace

extern "C" {

const char *gq_status_string(int status)
{
    switch (status) {
    case GQ_OK: return "GQ_OK";
    case GQ_ERR_NULL: return "GQ_ERR_NULL: a required pointer is NULL";
    case GQ_ERR_ALIGN: return "GQ_ERR_ALIGN: a pointer is not 16-byte aligned";
    case GQ_ERR_SHAPE: return "GQ_ERR_SHAPE: rows/K/M/k outside the legal range";
    case GQ_ERR_WORKSPACE: return "GQ_ERR_WORKSPACE: workspace missing or too small";
    case GQ_ERR_CUDA: return "GQ_ERR_CUDA: the CUDA runtime reported an error";
    case GQ_ERR_TIMEOUT: return "GQ_ERR_TIMEOUT: a bounded in-kernel wait gave up";
    case GQ_ERR_FORMAT: return "GQ_ERR_FORMAT: unknown block format";
    }
    return "unknown gq_status";
}

size_t gq_packed_bytes(int format, int rows, int K)
{
    if (!valid_format(format) || rows < 1 || K < block_weights(format) || K % block_weights(format) != 0)
        return 0;
    return static_cast<size_t>(rows) * static_cast<size_t>(K / block_weights(format)) *
           static_cast<size_t>(block_bytes(format));
}

static int pack_common(int format, const void *src, void *dst, int rows, int K, bool unpack, gq_stream_t s)
{
    if (!valid_format(format)) return GQ_ERR_FORMAT;
    if (!src || !dst) return GQ_ERR_NULL;
    if (!aligned16(src) || !aligned16(dst)) return GQ_ERR_ALIGN;
    if (gq_packed_bytes(format, rows, K) == 0) return GQ_ERR_SHAPE;
    return launch_pack(format, src, dst, rows, K, unpack, reinterpret_cast<cudaStream_t>(s));
}

int gq_pack(int format, const void *W_canon, void *W_packed, int rows, int K, gq_stream_t stream)
{
    return pack_common(format, W_canon, W_packed, rows, K, false, stream);
}

int gq_unpack(int format, const void *W_packed, void *W_canon, int rows, int K, gq_stream_t stream)
{
    return pack_common(format, W_packed, W_canon, rows, K, true, stream);
}

int gq_q4_0_matvec(const void *W, const float *x, float *y, int rows, int K, int M, gq_stream_t stream)
{
    int st = check_matvec(GQ_FORMAT_Q4_0, W, x, y, rows, K, M);
    if (st != GQ_OK) return st;
    // rows of whole 8-block groups stream through the shared-memory ring; other K take the register path
    if (ring_preferred(rows, K / 32) && ring_q4_0_supported(K / 32)) {
        st = launch_ring_q4_0(W, x, nullptr, nullptr, y, rows, K, reinterpret_cast<cudaStream_t>(stream));
        if (st != GQ_ERR_SHAPE) return st;
    }
    return launch_q4_0_matvec(W, x, y, rows, K, choose_matvec_geo(GQ_FORMAT_Q4_0, rows, K / 32, aligned32(W)),
                              reinterpret_cast<cudaStream_t>(stream));
}

int gq_q8_0_matvec(const void *W, const float *x, float *y, int rows, int K, int M, gq_stream_t stream)
{
    int st = check_matvec(GQ_FORMAT_Q8_0, W, x, y, rows, K, M);
    if (st != GQ_OK) return st;
    if (!aligned32(W)) return GQ_ERR_ALIGN;  // 32-byte weight loads
    return launch_q8_0_matvec(W, x, y, rows, K, choose_matvec_geo(GQ_FORMAT_Q8_0, rows, K / 32, false),
                              reinterpret_cast<cudaStream_t>(stream));
}

int gq_q4k_matvec(const void *W, const float *x, float *y, int rows, int K, int M, gq_stream_t stream)
{
    int st = check_matvec(GQ_FORMAT_Q4_K, W, x, y, rows, K, M);
    if (st != GQ_OK) return st;
    if (ring_preferred(rows, K / 32)) {
        st = launch_ring_q4k(W, x, y, rows, K, reinterpret_cast<cudaStream_t>(stream));
        if (st != GQ_ERR_SHAPE) return st;
    }
    return launch_q4k_matvec(W, x, y, rows, K, choose_matvec_geo(GQ_FORMAT_Q4_K, rows, K / 32, aligned32(W)),
                             reinterpret_cast<cudaStream_t>(stream));
}

int gq_q6k_matvec(const void *W, const float *x, float *y, int rows, int K, int M, gq_stream_t stream)
{
    int st = check_matvec(GQ_FORMAT_Q6_K, W, x, y, rows, K, M);
    if (st != GQ_OK) return st;
    return launch_q6k_matvec(W, x, y, rows, K, reinterpret_cast<cudaStream_t>(stream));
}

int gq_ffn_gate_up_gelu(const void *W_gate, const void *W_up, const float *x, float *h, int rows, int K,
                        int M, gq_stream_t stream)
{
    if (!W_up) return GQ_ERR_NULL;
    if (!aligned16(W_up)) return GQ_ERR_ALIGN;
    int st = check_matvec(GQ_FORMAT_Q4_0, W_gate, x, h, rows, K, M);
    if (st != GQ_OK) return st;
    if (ring_preferred(rows, K / 32) && ring_q4_0_supported(K / 32)) {
        st = launch_ring_ffn(W_gate, W_up, x, h, rows, K, reinterpret_cast<cudaStream_t>(stream));
        if (st != GQ_ERR_SHAPE) return st;
    }
    return launch_ffn_gate_up(W_gate, W_up, x, h, rows, K, choose_ffn_geo(rows, K / 32, aligned32(W_gate) && aligned32(W_up)),
                              reinterpret_cast<cudaStream_t>(stream));
}

int gq_q4_0_geglu_down(const void *W_down, const float *g, const float *u, float *y, int rows, int K, int M,
                       gq_stream_t stream)
{
    if (!u) return GQ_ERR_NULL;
    int st = check_matvec(GQ_FORMAT_Q4_0, W_down, g, y, rows, K, M);
    if (st != GQ_OK) return st;
    if (!aligned16(u)) return GQ_ERR_ALIGN;
    if (ring_preferred(rows, K / 32) && ring_q4_0_supported(K / 32)) {
        st = launch_ring_q4_0(W_down, nullptr, g, u, y, rows, K, reinterpret_cast<cudaStream_t>(stream));
        if (st != GQ_ERR_SHAPE) return st;
    }
    return launch_q4_0_geglu_down(W_down, g, u, y, rows, K,
                                  choose_matvec_geo(GQ_FORMAT_Q4_0, rows, K / 32, aligned32(W_down)),
                                  reinterpret_cast<cudaStream_t>(stream));
}

size_t gq_logits_topk_workspace_bytes(int rows, int K, int k)
{
    if (rows < 1 || k < 1 || k > GQ_MAX_TOPK) return 0;
    return logits_topk_ws_bytes(rows, K, k);
}

int gq_logits_topk(const void *W, const float *x, float softcap, int k, int *idx, float *val,
                   float *logits_or_null, void *workspace, size_t workspace_bytes, int rows, int K, int M,
                   gq_stream_t stream)
{
    int st = check_matvec(GQ_FORMAT_Q8_0, W, x, x, rows, K, M);
    if (st != GQ_OK) return st;
    if (!aligned32(W)) return GQ_ERR_ALIGN;  // 32-byte weight loads
    if (!idx || !val) return GQ_ERR_NULL;
    if (!aligned16(idx) || !aligned16(val) || (logits_or_null && !aligned16(logits_or_null)))
        return GQ_ERR_ALIGN;
    if (k < 1 || k > GQ_MAX_TOPK || k > rows) return GQ_ERR_SHAPE;
    if (!(softcap == softcap)) return GQ_ERR_SHAPE; /* NaN cap */
    if (!workspace) return GQ_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GQ_ERR_ALIGN;
    if (workspace_bytes < logits_topk_ws_bytes(rows, K, k)) return GQ_ERR_WORKSPACE;
    return launch_logits_topk(W, x, softcap, k, idx, val, logits_or_null, workspace, workspace_bytes, rows,
                              K, choose_logits_geo(rows, K / 32), reinterpret_cast<cudaStream_t>(stream));
}

int gq_quantize_q8_0(const float *X, int8_t *Xq, float *dx, int K, int M, gq_stream_t stream)
{
    if (!X || !Xq || !dx) return GQ_ERR_NULL;
    if (!aligned16(X) || !aligned16(Xq) || !aligned16(dx)) return GQ_ERR_ALIGN;
    if (M < 1 || K < 32 || K % 32 != 0) return GQ_ERR_SHAPE;
    return launch_quantize_q8_0(X, Xq, dx, K, M, reinterpret_cast<cudaStream_t>(stream));
}

int gq_rmsnorm_quantize_q8_0(const float *X, const float *w, float offset, float eps, int8_t *Xq, float *dx,
                             int K, int M, gq_stream_t stream)
{
    if (!X || !w || !Xq || !dx) return GQ_ERR_NULL;
    if (!aligned16(X) || !aligned16(w) || !aligned16(Xq) || !aligned16(dx)) return GQ_ERR_ALIGN;
    if (M < 1 || K < 32 || K % 32 != 0 || K > GQ_MAX_K) return GQ_ERR_SHAPE;
    if (!(eps > 0.0f) || !isfinite(eps) || !isfinite(offset)) return GQ_ERR_SHAPE;
    return launch_rmsnorm_q8_0(X, w, offset, eps, Xq, dx, K, M, reinterpret_cast<cudaStream_t>(stream));
}

int gq_rmsnorm_sum_squares(const float *X, double *ss, int K, int M, gq_stream_t stream)
{
    if (!X || !ss) return GQ_ERR_NULL;
    if (!aligned16(X) || !aligned16(ss)) return GQ_ERR_ALIGN;
    if (M < 1 || K < 32 || K % 32 != 0 || K > GQ_MAX_K) return GQ_ERR_SHAPE;
    return launch_row_sum_squares(X, ss, K, M, reinterpret_cast<cudaStream_t>(stream));
}

size_t gq_q4_0_gemm_workspace_bytes(int K, int M)
{
    // enough for every contraction path
    const size_t a = gemm_workspace_bytes(K, M), b = gemm_split_workspace_bytes(K, M),
                 c = gemm_mma_workspace_bytes(K, M);
    const size_t ab = a > b ? a : b;
    return ab > c ? ab : c;
}

int gq_q4_0_gemm_q8act(const void *W, const int8_t *Xq, const float *dx, float *Y, void *workspace,
                       size_t workspace_bytes, int rows, int K, int M, gq_stream_t stream)
{
    if (!W || !Xq || !dx || !Y || !workspace) return GQ_ERR_NULL;
    if (!aligned16(W) || !aligned16(Xq) || !aligned16(dx) || !aligned16(Y) || !aligned16(workspace))
        return GQ_ERR_ALIGN;
    if (rows < 1 || M < 1 || K < 32 || K % 32 != 0) return GQ_ERR_SHAPE;
    if (workspace_bytes < gq_q4_0_gemm_workspace_bytes(K, M)) return GQ_ERR_WORKSPACE;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // up to a few hundred tokens: exact block dots in registers (mma.sync)
    if (gemm_mma_supported(K, M) && M <= gemm_mma_max_tokens())
        return launch_gemm_mma(W, Xq, dx, Y, workspace, workspace_bytes, rows, K, M, st);
    // few tokens, other K: decode each weight once on the CUDA cores and apply it to every token
    if (gemm_small_supported(K, M)) return launch_gemm_small(W, Xq, dx, Y, rows, K, M, st);
    if (gemm_split_supported(K) && !gemm_force_block_path())
        return launch_gemm_split(W, Xq, dx, Y, workspace, workspace_bytes, rows, K, M, st);
    return launch_gemm_q8act_tc(W, Xq, dx, Y, workspace, workspace_bytes, rows, K, M, st);
}

int gq_q4_0_gemm_block_dots(const void *W, const int8_t *Xq, int32_t *D, void *workspace, size_t workspace_bytes,
                            int rows, int K, int M, gq_stream_t stream)
{
    if (!W || !Xq || !D || !workspace) return GQ_ERR_NULL;
    if (!aligned16(W) || !aligned16(Xq) || !aligned16(D) || !aligned16(workspace)) return GQ_ERR_ALIGN;
    if (rows < 1 || M < 1 || K < 32 || K % 32 != 0) return GQ_ERR_SHAPE;
    if (workspace_bytes < gq_q4_0_gemm_workspace_bytes(K, M)) return GQ_ERR_WORKSPACE;
    return launch_block_dots_tc(W, Xq, D, workspace, workspace_bytes, rows, K, M,
                                reinterpret_cast<cudaStream_t>(stream));
}

int gq_device_status(int reset) { return read_device_status(reset != 0); }

int gq_selftest_bounded_wait(gq_stream_t stream)
{
    return launch_selftest_bounded_wait(reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
