// GEMV kernels of one activation mode (activation codes staged by the separate quantiser).
#include "gemv_impl.cuh"

namespace qspec {
namespace gemv_impl {
QSPEC_GEMV_MODE_UNIT(1)
}  // namespace gemv_impl
}  // namespace qspec
