// GEMV kernels of one activation mode (W4A8).
#include "gemv_impl.cuh"

namespace qspec {
namespace gemv_impl {
QSPEC_GEMV_MODE_UNIT(8)
}  // namespace gemv_impl
}  // namespace qspec
