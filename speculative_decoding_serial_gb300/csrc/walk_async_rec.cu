// walk_async_rec.cu — walk kernel instantiations of the recurrent head that copy each step's base logits a step
// ahead (cp.async), for walks that read them from host memory in place.
#include "walk_launch.cuh"

namespace whead {
int launch_walk_async_recurrent(const WalkLaunch& l, const WalkArgs& a) { return launch_dispatch<true, true>(l, a); }
}  // namespace whead
