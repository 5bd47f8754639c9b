// lr_sel_f32_noz_sp.cu -- one compiled variant of the selective scan kernel:
// fp32 I/O, without a z gate, softplus applied to dt (see lr_selective.cuh).
#include "lr_selective.cuh"

namespace lr {
namespace sel {
LR_SEL_DEFINE(f32_noz_sp, float, true, false, true)
}  // namespace sel
}  // namespace lr
