// gq_geo.cu -- geometry choice for the matvec-family kernels.
//
// Chosen by measurement on GB300 (sweeps over lane-group width LG, rows per
// group R, loads in flight U, and blocks per lane load P at the workload
// shapes).  The 4-bit formats use P = 2 (32-byte loads of two consecutive
// blocks) whenever a row holds an even number of blocks and the weights are
// 32-byte aligned (measured: on par with or slightly ahead of 16-byte loads).
#include "gq_host.h"

namespace gq {

MatvecGeo choose_matvec_geo(int format, int rows, int nb, bool pair_ok)
{
    (void)rows;
    if (format == GQ_FORMAT_Q8_0) return MatvecGeo{16, 2, 4, 8, 1};
    if (pair_ok && nb % 2 == 0) return MatvecGeo{32, 2, nb >= 512 ? 4 : 2, 8, 2};
    return MatvecGeo{(nb % 32 == 0) ? 32 : 16, nb >= 512 ? 1 : 2, 4, 8, 1};
}

MatvecGeo choose_logits_geo(int rows, int nb)
{
    (void)rows;
    (void)nb;
    return MatvecGeo{8, 2, 4, 8, 1};
}

MatvecGeo choose_ffn_geo(int rows, int nb, bool pair_ok)
{
    (void)rows;
    if (pair_ok && nb % 2 == 0) return MatvecGeo{32, 2, 2, 8, 2};
    return MatvecGeo{(nb % 32 == 0) ? 32 : 16, 1, 4, 8, 1};
}

}  // namespace gq
