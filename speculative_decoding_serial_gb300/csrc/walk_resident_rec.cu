// walk_resident_rec.cu — walk kernel instantiations of the recurrent head for base logits read at each step.
#include "walk_launch.cuh"

namespace whead {
int launch_walk_resident_recurrent(const WalkLaunch& l, const WalkArgs& a) { return launch_dispatch<false, true>(l, a); }
}  // namespace whead
