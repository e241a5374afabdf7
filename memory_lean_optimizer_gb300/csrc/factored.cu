// factored.cu -- factored second-moment step (placeholder until the kernels land).
#include "factored.h"

namespace lmo {
struct FactoredPlan { int unused; };
int factored_plan_build(FactoredPlan*& plan, const std::vector<optim_tensor_desc_t>&) {
    plan = nullptr;
    return set_error(OPTIM_EINVAL, "factored groups are not available in this build");
}
void factored_plan_free(FactoredPlan*& plan) { delete plan; plan = nullptr; }
int launch_factored_step(const FactoredPlan*, const uint16_t* const*, const FactoredScalars&, cudaStream_t, cudaEvent_t) {
    return set_error(OPTIM_EINVAL, "factored groups are not available in this build");
}
}  // namespace lmo
