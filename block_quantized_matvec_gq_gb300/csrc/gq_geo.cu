// gq_geo.cu -- geometry choice for the matvec-family kernels.
//
// Chosen by measurement on GB300 (a sweep over lane-group width LG, rows per
// group R and blocks in flight U at the workload shapes): U = 4 wins for
// every format; 16- or 32-lane groups beat 8-lane groups for the 4-bit
// formats; the tied-logit kernel prefers 8-lane groups of 2 rows.
#include "gq_host.h"

namespace gq {

MatvecGeo choose_matvec_geo(int format, int rows, int nb)
{
    (void)rows;
    const int lg_wide = (nb % 32 == 0) ? 32 : 16;
    switch (format) {
    case GQ_FORMAT_Q8_0: return MatvecGeo{16, 2, 4, 8};
    case GQ_FORMAT_Q4_0:
    case GQ_FORMAT_Q4_K:
    default: return MatvecGeo{lg_wide, nb >= 512 ? 1 : 2, 4, 8};
    }
}

MatvecGeo choose_logits_geo(int rows, int nb)
{
    (void)rows;
    (void)nb;
    return MatvecGeo{8, 2, 4, 8};
}

MatvecGeo choose_ffn_geo(int rows, int nb)
{
    (void)rows;
    return MatvecGeo{(nb % 32 == 0) ? 32 : 16, 1, 4, 8};
}

}  // namespace gq
