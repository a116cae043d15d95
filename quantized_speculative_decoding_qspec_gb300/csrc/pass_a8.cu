// Linear-pass kernels of one activation mode (W4A8).
#include "pass_impl.cuh"

namespace qspec {
namespace pass_impl {
QSPEC_PASS_MODE_UNIT(8)
}  // namespace pass_impl
}  // namespace qspec
