// The multi-query split kernel and its combine for INT8 caches (the kernel
// templates are in mq_split.cuh), compiled apart from mq.cu so the two build
// in parallel.
#include "mq_split.cuh"

namespace pkv {

bool mq_pick_i8(pkv_dtype q_dtype, int D, int G, int nw, MqOps* o) {
    if (q_dtype == PKV_BF16) return mq_pick_d<I8, BF16>(D, G, nw, o);
    if (q_dtype == PKV_F16) return mq_pick_d<I8, F16>(D, G, nw, o);
    return false;
}

}  // namespace pkv
