// walk_async.cu — walk kernel instantiations of the Markov head that copy each step's base logits a step ahead
// (cp.async), for walks that read them from host memory in place.
#include "walk_launch.cuh"

namespace whead {
int launch_walk_async_markov(const WalkLaunch& l, const WalkArgs& a) { return launch_dispatch<true, false>(l, a); }
}  // namespace whead
