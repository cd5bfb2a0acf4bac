// walk_resident.cu — walk kernel instantiations for base logits read at each step (device memory).
#include "walk_launch.cuh"

namespace whead {
int launch_walk_resident(const WalkLaunch& l, const WalkArgs& a) { return launch_dispatch<false>(l, a); }
}  // namespace whead
