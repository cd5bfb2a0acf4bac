// walk_launch.h — launching one walk: the interface between the host library (whead_api.cu) and the
// translation units that hold the walk kernel's instantiations (walk_resident.cu, walk_async.cu), which are
// compiled in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace whead {

struct WalkArgs;

// Where and how one walk runs. tmap / tmap128: W's tensor maps (16- and 128-row boxes). smem_bytes: the
// plan's dynamic shared memory; the launcher adds the incoming base-logit buffer when the walk copies base
// logits asynchronously (kFlagBaseAsync in the arguments' flags). r and nh (batch halves: B <= 8 nh) and f8
// select the kernel instantiation.
struct WalkLaunch {
  const CUtensorMap* tmap;
  const CUtensorMap* tmap128;
  cudaStream_t stream;
  int smem_optin;
  int grid;
  int smem_bytes;
  int r;
  int nh;
  bool f8;
};

// Cooperative launch of the walk kernel; WHEAD_OK, WHEAD_ERR_NO_COOP (grid not co-resident),
// WHEAD_ERR_UNSUPPORTED (no instantiation for r / f8) or WHEAD_ERR_CUDA. The Markov and recurrent heads have
// instantiations of their own, in translation units of their own (compiled in parallel).
int launch_walk_resident_markov(const WalkLaunch& l, const WalkArgs& a);     // base logits read at each step
int launch_walk_resident_recurrent(const WalkLaunch& l, const WalkArgs& a);
int launch_walk_async_markov(const WalkLaunch& l, const WalkArgs& a);        // base logits copied a step ahead
int launch_walk_async_recurrent(const WalkLaunch& l, const WalkArgs& a);

}  // namespace whead
