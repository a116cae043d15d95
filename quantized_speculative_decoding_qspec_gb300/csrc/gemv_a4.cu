// GEMV kernels of one activation mode (W4A4).
#include "gemv_impl.cuh"

namespace qspec {
namespace gemv_impl {
QSPEC_GEMV_MODE_UNIT(4)
}  // namespace gemv_impl
}  // namespace qspec
