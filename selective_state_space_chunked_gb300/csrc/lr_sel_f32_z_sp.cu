// lr_sel_f32_z_sp.cu -- one compiled variant of the selective scan kernel:
// fp32 I/O, with the silu(z) gate, softplus applied to dt (see lr_selective.cuh).
#include "lr_selective.cuh"

namespace lr {
namespace sel {
LR_SEL_DEFINE(f32_z_sp, float, true, true, true)
}  // namespace sel
}  // namespace lr
