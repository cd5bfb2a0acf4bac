// walk_async.cu — walk kernel instantiations that copy each step's base logits a step ahead (cp.async), for
// walks that read them from host memory in place.
#include "walk_launch.cuh"

namespace whead {
int launch_walk_async(const WalkLaunch& l, const WalkArgs& a) { return launch_dispatch<true>(l, a); }
}  // namespace whead
