// Instantiations of the dequantising tensor-core W4A16 kernel (dq_impl.cuh).
#include "dq_impl.cuh"

namespace qspec {

qspec_status dq_launch(int NM, int J, const CUtensorMap& tmW, const CUtensorMap& tmX, const dq::DqArgs& args, int P,
                       cudaStream_t stream) {
  if (NM == 128) {
    if (J == 1) return dq::launch<128, 1>(tmW, tmX, args, P, stream);
    if (J == 2) return dq::launch<128, 2>(tmW, tmX, args, P, stream);
    return QSPEC_ERR_UNSUPPORTED_SHAPE;
  }
  if (NM == 256 && J == 1) return dq::launch<256, 1>(tmW, tmX, args, P, stream);
  return QSPEC_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace qspec
