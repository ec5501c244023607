// tc.cu -- placeholder; replaced by the tcgen05 path.
#include "internal.h"
namespace conv_epi {
conv_epi_status tc_supported(const conv_epi_desc &, const conv_epi_epilogue_desc *) { return CONV_EPI_ERR_UNSUPPORTED; }
size_t tc_wpack_bytes(const conv_epi_desc &) { return 256; }
int tc_gn_units(const conv_epi_desc &, int, int) { return 1; }
conv_epi_status tc_forward(conv_epi_handle, const float *, const float *, const float *,
                           const conv_epi_epilogue_desc &, float *, cudaStream_t) { return CONV_EPI_ERR_UNSUPPORTED; }
}  // namespace conv_epi
