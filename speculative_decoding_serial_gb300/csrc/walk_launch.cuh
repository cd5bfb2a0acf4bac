// walk_launch.cuh — the kernel instantiations behind launch_walk_resident / launch_walk_async (included by
// walk_resident.cu and walk_async.cu only).
#pragma once

#include "../../include/whead.h"
#include "walk_kernel.cuh"
#include "walk_launch.h"

namespace whead {
namespace {

template <int KB, int NH, bool NB1, bool F8, bool ASYNC, bool REC>
int launch_t(const WalkLaunch& l, const WalkArgs& a) {
  auto fn = walk_kernel<KB, NH, NB1, F8, ASYNC, REC>;
  static int attr_bytes = 0;  // largest dynamic shared memory size granted so far (per instantiation)
  const int smem = l.smem_bytes + ((a.flags & kFlagBaseAsync) ? base_in_bytes(a.B, a.ng) : 0);
  if (smem > attr_bytes) {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, l.smem_optin) != cudaSuccess)
      return WHEAD_ERR_CUDA;
    attr_bytes = l.smem_optin;
  }
  void* args[] = {(void*)l.tmap, (void*)l.tmap128, (void*)&a};
  cudaError_t e = cudaLaunchCooperativeKernel((const void*)fn, dim3(l.grid), dim3(kThreads), args, (size_t)smem,
                                              l.stream);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    (void)cudaGetLastError();
    return WHEAD_ERR_NO_COOP;
  }
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return WHEAD_ERR_CUDA;
  }
  return WHEAD_OK;
}

// Instantiation for (rank boxes KB = r / 64, batch halves, single walk, E4M3 weights) of one head kind.
template <bool ASYNC, bool REC>
int launch_dispatch(const WalkLaunch& l, const WalkArgs& a) {
  const bool one = a.B == 1;
  if (l.f8) {  // E4M3 weights: 128 codes per box, one batch half (at most 4 walks), r = 128 or 256
    switch ((l.r / 128) * 2 + (one ? 1 : 0)) {
      case 2: return launch_t<1, 1, false, true, ASYNC, REC>(l, a);
      case 3: return launch_t<1, 1, true, true, ASYNC, REC>(l, a);
      case 4: return launch_t<2, 1, false, true, ASYNC, REC>(l, a);
      case 5: return launch_t<2, 1, true, true, ASYNC, REC>(l, a);
      default: return WHEAD_ERR_UNSUPPORTED;
    }
  }
  switch ((l.r / 64) * 4 + (l.nh - 1) * 2 + (one ? 1 : 0)) {
    case 4: return launch_t<1, 1, false, false, ASYNC, REC>(l, a);
    case 5: return launch_t<1, 1, true, false, ASYNC, REC>(l, a);
    case 6: return launch_t<1, 2, false, false, ASYNC, REC>(l, a);
    case 8: return launch_t<2, 1, false, false, ASYNC, REC>(l, a);
    case 9: return launch_t<2, 1, true, false, ASYNC, REC>(l, a);
    case 10: return launch_t<2, 2, false, false, ASYNC, REC>(l, a);
    case 12: return launch_t<3, 1, false, false, ASYNC, REC>(l, a);
    case 13: return launch_t<3, 1, true, false, ASYNC, REC>(l, a);
    case 14: return launch_t<3, 2, false, false, ASYNC, REC>(l, a);
    case 16: return launch_t<4, 1, false, false, ASYNC, REC>(l, a);
    case 17: return launch_t<4, 1, true, false, ASYNC, REC>(l, a);
    case 18: return launch_t<4, 2, false, false, ASYNC, REC>(l, a);
    default: return WHEAD_ERR_UNSUPPORTED;
  }
}

}  // namespace
}  // namespace whead
