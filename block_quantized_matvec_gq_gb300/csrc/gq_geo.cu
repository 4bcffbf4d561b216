// gq_geo.cu -- geometry choice for the matvec-family kernels.
//
// Chosen by measurement on GB300 (sweeps over lane-group width LG, rows per
// group R, loads in flight U, and blocks per lane load P at the workload
// shapes).  With the register-lean 4-bit core, 16-byte loads (P = 1) beat
// the 32-byte block-pair loads at every measured shape; LG = 32 when a row's
// block count is a multiple of 32, else 16 (less idle lanes in the last
// step); U = 2 (with the balanced K-split schedule, two loads in flight
// also beat four on the 5376 x 21504 down projection: 20.6 vs 22.0 us).
#include "gq_host.h"

namespace gq {

MatvecGeo choose_matvec_geo(int format, int rows, int nb, bool pair_ok)
{
    (void)rows;
    (void)pair_ok;
    if (format == GQ_FORMAT_Q8_0) return MatvecGeo{16, 2, 4, 8, 1};
    return MatvecGeo{(nb % 32 == 0) ? 32 : 16, 2, 2, 8, 1};
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
    (void)nb;
    (void)pair_ok;
    return MatvecGeo{8, 1, 4, 8, 1};
}

}  // namespace gq
