// scan_fwd_tma_f32.cu -- the fp32-I/O instances of the TMA forward scan (scan_fwd_tma.cuh); a
// translation unit of their own so that the two I/O types compile in parallel.
#include "scan_fwd_tma.cuh"

namespace ssm {

#define SSM_INSTANTIATE_F32(NS, TPC, SA, THR, CK) \
  template cudaError_t launch_fwd_tma_t<float, NS, TPC, SA, THR, CK>(FwdTmaArgs&, size_t, size_t, cudaStream_t);
SSM_FWD_TMA_VARIANTS(SSM_INSTANTIATE_F32)
#undef SSM_INSTANTIATE_F32

}  // namespace ssm
