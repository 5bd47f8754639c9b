// lr_sel_bf16_noz_nosp.cu -- one compiled variant of the selective scan kernel:
// bf16 I/O, without a z gate, dt taken as delta (see lr_selective.cuh).
#include "lr_selective.cuh"

namespace lr {
namespace sel {
LR_SEL_DEFINE(bf16_noz_nosp, __nv_bfloat16, false, false, false)
}  // namespace sel
}  // namespace lr
