// walk_resident.cu — walk kernel instantiations of the Markov head for base logits read at each step.
#include "walk_launch.cuh"

namespace whead {
int launch_walk_resident_markov(const WalkLaunch& l, const WalkArgs& a) { return launch_dispatch<false, false>(l, a); }
}  // namespace whead
