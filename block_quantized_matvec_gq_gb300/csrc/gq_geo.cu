// gq_geo.cu -- geometry choice for the matvec-family kernels.
//
// Chosen by measurement on GB300 (sweeps over lane-group width LG, rows per
// group R and blocks per batch U at the workload shapes).  The 4-bit
// streams load a batch of U blocks of every row before computing it:
// LG = 32 when a row's block count is a multiple of 32, else 16 (fewer idle
// lanes in the last step), R = 2, U = 4 (21504 x 5376 Q4_K: 21.3 us, against
// 22.0 with LG 8 and 28-29 with eight-block batches; the 4096 x 4096 Q4_0:
// 3.8 us).  The FFN pair: LG = 16, R = 1, U = 4 (two matrices per row).
#include <stdio.h>
#include <stdlib.h>

#include "gq_host.h"

namespace gq {

#ifdef GQ_TUNING
// Geometry sweeps: a tuning build reads overrides from the environment.
static MatvecGeo tuned(const char *prefix, MatvecGeo g)
{
    char name[64];
    const char *v;
    snprintf(name, sizeof name, "%s_LG", prefix);
    if ((v = getenv(name))) g.lg = atoi(v);
    snprintf(name, sizeof name, "%s_R", prefix);
    if ((v = getenv(name))) g.r = atoi(v);
    snprintf(name, sizeof name, "%s_U", prefix);
    if ((v = getenv(name))) g.u = atoi(v);
    return g;
}
static int ring_override()
{
    const char *v = getenv("GQ_RING");
    return v ? atoi(v) : -1;
}
bool gemm_force_block_path()
{
    const char *v = getenv("GQ_GEMM_BLOCK");
    return v && atoi(v) != 0;
}
#else
static MatvecGeo tuned(const char *, MatvecGeo g) { return g; }
static int ring_override() { return -1; }
bool gemm_force_block_path() { return false; }
#endif

// Register-stream schedule from tasks per resident warp: <= 1.25 balanced
// with the first loads issued early (mode 2); < 1.75 balanced (mode 1) on
// rows of at least 512 blocks, whose leftover rows split along K into eight
// slices that still fill the lanes; else round-robin (mode 0).  Measured on
// Q4_0 between 1.25 and 1.75 tasks per warp: at K = 21504 balanced 25.5 /
// 27.6 / 31.1 us against 27.8 / 30.6 / 30.6 round-robin (6400 / 7296 / 8192
// rows); at K = 5376 round-robin 14.9 / 15.3 / 15.7 against 14.8 / 16.5 /
// 19.4 (12800 / 14592 / 16384 rows); at K = 4096 round-robin 6.5 / 6.8 / 6.9
// against 7.9 / 9.5 / 11.8 (6144 / 7168 / 8192 rows).
int schedule_mode(long long ntasks, long long warps, int nb)
{
#ifdef GQ_TUNING
    if (const char *v = getenv("GQ_MODE")) return atoi(v);
#endif
    if (ntasks * 4 <= warps * 5) return 2;
    if (ntasks * 4 < warps * 7) return nb >= 512 ? 1 : 0;
    return 0;
}

// Short, wide matrices (fewer than eight rows per SM) of rows longer than 128
// blocks take the shared-memory ring (with a cluster split-K below four rows
// per SM): the register streams would leave most SMs idle, since their grid
// holds one CTA per eight row tasks.  Measured on Q4_0: 256 x 21504 in 5.1
// instead of 13.6 us, 8 x 49152 in 3.8 instead of 17.9 us; 64 to 512 rows of
// 5376 in 4.0-4.3 instead of 4.9-5.0 us; 608 / 768 / 1024 rows of 5376 in
// 3.6 / 3.8 / 3.9 against 5.0 / 5.1 / 5.1 us, of 21504 in 6.0 / 8.0 / 8.2
// against 10.5 / 10.5 / 10.6 us, of 8192 in 3.9 / 4.0 / 4.1 against 4.0 / 4.0
// / 4.2 us.  At 1536 rows the streams are level or ahead (5376: 5.2 against
// 5.5 us).  At 4096 (128 blocks) the streams are faster at every row count
// (64 to 512 rows: 2.3 against 4.0-4.1 us; 1024: 2.4 against 3.5).  Q4_K
// at 608 / 1024 / 1215 rows: 3.9 / 4.1 / 4.3 against 6.2 / 6.3 / 12.0 us
// (K = 5376), 6.4 / 8.8 / 9.0 against 13.6 / 14.0 / 18.0 us (K = 21504).
bool ring_preferred(int rows, int nb)
{
    const int o = ring_override();
    if (o >= 0) return o != 0;
    return rows < 8 * sm_count() && nb > 128;
}

// 4-bit streams: 32 lanes per row group (2-row tasks) when the row length is
// a multiple of 32 blocks, else 16 (4-row tasks).  Q4_0 rows shorter than 512
// blocks that would leave 32-lane tasks at 1.25 to 1.75 per resident warp
// take 16 lanes instead: half as many tasks fit one balanced round, where
// the 32-lane tasks would run round-robin with a sparse second round.
// Measured on Q4_0 (us per step, 32 lanes against 16): K = 4096, 6144 rows
// 6.55 / 5.85, 8192 rows 6.89 / 6.08; K = 8192, 8192 rows 11.6 / 11.2;
// K = 14336, 8192 rows 20.4 / 19.8.  Outside that band 32 lanes win (4096 x
// 4096 3.77 / 4.36, 12288 x 4096 9.34 / 10.9, 4096 x 8192 6.31 / 7.94,
// 7296 x 21504 27.5 / 30.1).
MatvecGeo choose_matvec_geo(int format, int rows, int nb, bool pair_ok)
{
    (void)pair_ok;
    if (format == GQ_FORMAT_Q8_0) return tuned("GQ_Q8", MatvecGeo{16, 2, 4, 8});
    int lg = (nb % 32 == 0) ? 32 : 16;
    if (lg == 32 && format == GQ_FORMAT_Q4_0 && nb < 512) {
        const long long tasks = (static_cast<long long>(rows) + 1) / 2;
        // resident warps: two CTAs of 256 threads per SM
        const long long warps = static_cast<long long>(sm_count()) * 16;
        if (tasks * 4 > warps * 5 && tasks * 4 <= warps * 7) lg = 16;
    }
    return tuned("GQ_Q4", MatvecGeo{lg, 2, 4, 8});
}

MatvecGeo choose_logits_geo(int rows, int nb)
{
    (void)rows;
    (void)nb;
    return tuned("GQ_LOG", MatvecGeo{8, 2, 4, 8});
}

// Largest token batch that takes the register-operand contraction
// (gq_gemm_mma.cu) rather than the tensor-memory tiles.  Measured on 21504 x
// 5376 weights: 103 us at M = 96 against 127 us on the tiles (which take the
// same time at any M <= 128); at M = 128 the tiles win (129 us).
int gemm_mma_max_tokens()
{
#ifdef GQ_TUNING
    if (const char *v = getenv("GQ_MMA_MAX")) return atoi(v);
#endif
    return 112;
}

MatvecGeo choose_q6k_geo() { return tuned("GQ_Q6", MatvecGeo{16, 2, 4, 8}); }

MatvecGeo choose_ffn_geo(int rows, int nb, bool pair_ok)
{
    (void)rows;
    (void)nb;
    (void)pair_ok;
    return tuned("GQ_FFN", MatvecGeo{16, 1, 4, 8});
}

}  // namespace gq
