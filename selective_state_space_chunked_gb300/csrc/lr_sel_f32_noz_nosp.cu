// lr_sel_f32_noz_nosp.cu -- one compiled variant of the selective scan kernel:
// fp32 I/O, without a z gate, dt taken as delta (see lr_selective.cuh).
#include "lr_selective.cuh"

namespace lr {
namespace sel {
LR_SEL_DEFINE(f32_noz_nosp, float, true, false, false)
}  // namespace sel
}  // namespace lr
