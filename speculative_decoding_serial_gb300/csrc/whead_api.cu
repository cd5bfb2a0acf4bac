// whead_api.cu — C ABI, placement planner and launch of the walk-resident serial draft head.
//
// "Weights That Stay: On-Chip Megakernels for Serial Heads in Speculative Decoding", Fig. 1: full or
// partial residency of W across the GPU's memory tiers. The planner below splits W into 16-row groups,
// gives each SM an equal run of groups and places them in shared memory, tensor memory and registers.
#include "../../include/whead.h"
#include "walk_kernel.cuh"
#include "walk_launch.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstring>
#include <new>

using namespace whead;

namespace {

struct Plan {
  bool ok = false;
  int G = 0, ng = 0, n_smem = 0, n_tmem = 0, n_rf = 0, n_stream = 0;
  uint32_t tmem_cols = 0;
  int smem_bytes = 0, smem_w_bytes = 0, ra = 0, Bcap = 0;
  uint32_t rf_warp_mask = 0;
  int ah_warp = 0;  // recurrent: the warp that computes the CTA's slice of A h each step
  int32_t wl_count[kWarps] = {};
  uint32_t wl[kWarps][kMaxWarpGroups] = {};
};

struct Scratch {
  unsigned long long* slots;  // [2 call parities][2 step parities] x sm_count x kMaxB words (walk-major per call)
  unsigned int* cnt;          // two counters, 128 bytes apart
  unsigned long long* ah;     // [2 call parities][2 step parities][kMaxB][r] tagged words
  int* status;
};

}  // namespace

struct whead_s {
  int device = 0;
  cudaStream_t stream = nullptr;
  whead_params p{};
  const uint16_t* W = nullptr;
  const uint16_t* E = nullptr;
  bool f8 = false;         // E4M3 weights: the handle's quantized copy of W and its row scales
  uint8_t* wq = nullptr;   // V x r E4M3 codes
  float* sw = nullptr;     // V row scales
  CUtensorMap tmap{};     // W: 64 x 16 boxes
  CUtensorMap tmap128{};  // W: 64 x 128 boxes
  int sm_count = 0, smem_optin = 0;
  int64_t slots_per_parity = 0;  // 2 step parities x sm_count x kMaxB words
  Plan plan[2];  // walks <= 8, walks <= 16
  void* scratch_block = nullptr;
  Scratch s{};
  uint32_t parity = 0;
  unsigned long long* trace = nullptr;
  int64_t trace_bytes = 0;
  // host-call staging (d_base only for base logits the GPU cannot read in place) and the status read-back
  int pageable_access = 0;  // the GPU reads any host memory through the host's page tables
  int* h_status = nullptr;  // pinned
  float* d_base = nullptr;
  float* d_u0 = nullptr;
  int32_t* d_tok = nullptr;
  void* d_logits = nullptr;
};

namespace {

// 128-byte boxes per row of W: 64 bf16 values, or 128 E4M3 codes
int kb_of(int r, bool f8 = false) { return f8 ? r / 128 : r / 64; }

// Planner: number of CTAs, groups per CTA and their tier; per-warp work lists balanced over the four
// SM sub-partitions (warp % 4), which each own one tensor core and one quarter of tensor memory.
// cap_*: most groups per CTA a tier may take (INT_MAX: as many as fit). fixed_tiers: the caps come from the
// caller (a measurement mode), so the grid is all SMs (or grid_req) and the groups past the caps are streamed.
Plan make_plan(int64_t V, int r, int kind, int Bcap, int NH, int sm_count, int smem_optin, int grid_req,
               int cap_smem = INT_MAX, int cap_tmem = INT_MAX, int cap_rf = INT_MAX, bool fixed_tiers = false,
               bool f8 = false) {
  Plan P;
  sm_count = std::min(sm_count, kMaxGrid);
  const int KB = kb_of(r, f8);
  const int64_t ngt = (V + kGroupRows - 1) / kGroupRows;
  const int64_t group_bytes = (int64_t)KB * kBoxBytes;
  const bool recurrent = kind == WHEAD_RECURRENT;
  // tensor-memory groups: 16 KB columns each, four lane quadrants side by side, within the 512 columns of one
  // allocation (ceil(n / 4) * 16 * KB <= 512)
  const int tmem_max = 4 * (32 / KB);
  const int rf_max = (NH == 1) ? 8 : 0;  // at most two register warps per lane quadrant

  auto fits = [&](int G, Plan& out, bool allow_stream) -> bool {
    const int64_t ng64 = (ngt + G - 1) / G;
    if (ng64 > 255) return false;
    const int ng = (int)ng64;
    const int ra = recurrent ? (r + G - 1) / G : 0;
    const SmemLayout L0 = SmemLayout::make(0, Bcap, r, ra, recurrent, ng, f8);
    const int64_t fixed = 1024 + L0.total;
    if (fixed > smem_optin) return false;  // e.g. a recurrent head's rows of A on too few CTAs: more CTAs are needed
    const int64_t smem_groups_max = std::min<int64_t>(cap_smem, std::max<int64_t>(0, (smem_optin - fixed) / group_bytes));
    int n_smem = (int)std::min<int64_t>(ng, smem_groups_max);
    int rem = ng - n_smem;
    int n_tmem = std::min(rem, std::min(tmem_max, cap_tmem));
    rem -= n_tmem;
    int n_rf = std::min(rem, std::min(rf_max, cap_rf));
    rem -= n_rf;
    if (rem > 0 && !allow_stream) return false;
    const int n_stream = rem;
    out = Plan();
    out.G = G;
    out.ng = ng;
    out.n_smem = n_smem;
    out.n_tmem = n_tmem;
    out.n_rf = n_rf;
    out.n_stream = n_stream;
    out.ra = ra;
    out.Bcap = Bcap;
    out.smem_w_bytes = (int)(n_smem * group_bytes);
    out.smem_bytes = (int)(1024 + SmemLayout::make(out.smem_w_bytes, Bcap, r, ra, recurrent, ng, f8).total);
    if (n_tmem > 0) {
      const int cols = ((n_tmem - 1) / 4 + 1) * 16 * KB;
      uint32_t pw = 32;
      while ((int)pw < cols) pw <<= 1;
      out.tmem_cols = pw;
    }
    // work lists. Warp roles per lane quadrant q (warps q, q + 4, q + 8): the highest warps of a quadrant
    // keep register-resident groups (one each), the rest own the quadrant's tensor-memory groups.
    const int rf_per_q = (n_rf + 3) / 4;
    const int tmem_warps_per_q = (kWarps / 4) - rf_per_q;
    if (n_tmem > 0 && tmem_warps_per_q < 1) return false;
    // relative cost of a group by tier, measured on GB300: tensor memory 5, register 5, shared 6, streamed 9. A
    // register warp runs its shared-memory groups slower (its resident group leaves fewer registers for loads in
    // flight): 8 there.
    int load[kWarps] = {};
    int sp_load[4] = {};
    auto push = [&](int w, uint32_t entry, int cost) -> bool {
      if (out.wl_count[w] >= kMaxWarpGroups) return false;
      out.wl[w][out.wl_count[w]++] = entry;
      load[w] += cost;
      sp_load[w & 3] += cost;
      return true;
    };
    for (int i = 0; i < n_rf; ++i) {
      const int q = i & 3, k = i >> 2;  // k-th register warp of quadrant q, counted from the top
      const int w = q + 4 * ((kWarps / 4) - 1 - k);  // never warp 0: it runs the exchange
      out.rf_warp_mask |= 1u << w;
      if (!push(w, wl_entry(n_smem + n_tmem + i, kTierRf, 0), 5)) return false;
    }
    for (int i = 0; i < n_tmem; ++i) {
      const int q = i & 3, idx = i >> 2;
      const int w = q + 4 * (idx % tmem_warps_per_q);
      if (!push(w, wl_entry(n_smem + i, kTierTmem, idx * 16 * KB), 5)) return false;
    }
    // least-loaded sub-partition, then its warp with the least load after the group (cost_rf on register warps)
    auto place = [&](uint32_t entry, int cost, bool rf_ok, int cost_rf) -> bool {
      auto cost_on = [&](int w) { return ((out.rf_warp_mask >> w) & 1u) ? cost_rf : cost; };
      int bq = -1, bw = -1;
      for (int q = 0; q < 4; ++q) {
        int w_best = -1;
        for (int w = q; w < kWarps; w += 4)
          if ((rf_ok || !((out.rf_warp_mask >> w) & 1u)) &&
              (w_best < 0 || load[w] + cost_on(w) < load[w_best] + cost_on(w_best)))
            w_best = w;
        if (w_best >= 0 && (bq < 0 || sp_load[q] < sp_load[bq])) {
          bq = q;
          bw = w_best;
        }
      }
      return bw >= 0 && push(bw, entry, cost_on(bw));
    };
    for (int i = 0; i < n_stream; ++i)
      if (!place(wl_entry(n_smem + n_tmem + n_rf + i, kTierStream, 0), 9, true, 9)) return false;
    for (int j = 0; j < n_smem; ++j)
      if (!place(wl_entry(j, kTierSmem, 0), 6, true, 8)) return false;
    // recurrent: the slice of A h goes to the least-loaded warp that keeps no register group (the register warps'
    // copy of the step loop does not carry that code)
    if (recurrent) {
      out.ah_warp = 0;
      for (int w = 1; w < kWarps; ++w)
        if (!((out.rf_warp_mask >> w) & 1u) && load[w] < load[out.ah_warp]) out.ah_warp = w;
    }
    out.ok = true;
    return true;
  };

  int G;
  if (fixed_tiers) {
    G = grid_req > 0 ? std::min(grid_req, sm_count) : sm_count;
    if (!fits(G, P, true)) P.ok = false;
    return P;
  }
  if (grid_req > 0) {
    G = std::min(grid_req, sm_count);
    if (!fits(G, P, true)) P.ok = false;
    return P;
  }
  // few CTAs for small heads (cheaper exchange), more until the shard fits on chip; if it never fits, all
  // SMs with the overflow streamed (partial residency)
  const int64_t target = 96 * 1024;
  G = (int)std::min<int64_t>(sm_count, std::max<int64_t>(1, (ngt * group_bytes + target - 1) / target));
  for (; G <= sm_count; ++G)
    if (fits(G, P, false)) return P;
  if (fits(sm_count, P, true)) return P;
  P.ok = false;
  return P;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

int launch(whead_t* h, const Plan& pl, const WalkArgs& a, int NH) {
  const WalkLaunch l{&h->tmap, &h->tmap128, h->stream, h->smem_optin, pl.G, pl.smem_bytes, h->p.r, NH, h->f8};
  if (a.kind == WHEAD_RECURRENT)
    return (a.flags & kFlagBaseAsync) ? launch_walk_async_recurrent(l, a) : launch_walk_resident_recurrent(l, a);
  return (a.flags & kFlagBaseAsync) ? launch_walk_async_markov(l, a) : launch_walk_resident_markov(l, a);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tagged A h words of one call parity: two step parities of up to kMaxB walks.
size_t ah_words_per_parity(int r) { return 2 * (size_t)kMaxB * r; }

// The next state of B walks for given winners x (global rows of E), one warp per (walk, element): Markov
// s_next[b] = E[x_b] (bf16 to fp32); recurrent s_next[b][i] = tanh(A[i,:] . s[b] + E[x_b, i] + c[i]) with the
// walk kernel's own order of operations (lane-strided fmaf, then a butterfly sum). A winner outside E gives a
// zero state and the status word WHEAD_ERR_INTERNAL.
__global__ void advance_kernel(int kind, const uint16_t* __restrict__ E, const float* __restrict__ A,
                               const float* __restrict__ c, const int32_t* __restrict__ x, const float* __restrict__ s,
                               float* __restrict__ s_next, int B, int r, int64_t e_rows, int* status) {
  const int wi = (int)(blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32), lane = threadIdx.x & 31;
  if (wi >= B * r) return;  // the same for every lane of the warp
  const int b = wi / r, i = wi % r;
  const int64_t xb = x[b];
  if (xb < 0 || xb >= e_rows) {
    if (lane == 0) {
      s_next[(int64_t)b * r + i] = 0.f;
      atomicCAS(status, 0, kStatusInternal);
    }
    return;
  }
  const float e = __uint_as_float((uint32_t)E[xb * r + i] << 16);
  if (kind == WHEAD_MARKOV) {
    if (lane == 0) s_next[(int64_t)b * r + i] = e;
    return;
  }
  float acc = 0.f;
  for (int k = lane; k < r; k += 32) acc = fmaf(A[(int64_t)i * r + k], s[(int64_t)b * r + k], acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    float pre = __fadd_rn(acc, e);
    if (c) pre = __fadd_rn(pre, c[i]);
    s_next[(int64_t)b * r + i] = tanhf(pre);
  }
}

// E4M3 weights: one warp per row quantizes it as a vector (scale max|w| / 448, codes E4M3(w / s)) with the
// same warp routine the walk uses for its state. EPL = r / 32 elements per lane.
template <int EPL>
__global__ void quantize_w_e4m3_kernel(const uint16_t* __restrict__ W, int64_t V, int r, uint8_t* __restrict__ Wq,
                                       float* __restrict__ sw) {
  const int lane = threadIdx.x & 31;
  const int64_t v = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (v >= V) return;  // the same for every lane of the warp
  const uint16_t* row = W + v * r + lane * EPL;
  uint32_t u[EPL / 2];
  if constexpr (EPL == 8) {
    const uint4 t = *reinterpret_cast<const uint4*>(row);
    u[0] = t.x; u[1] = t.y; u[2] = t.z; u[3] = t.w;
  } else {
    const uint2 t = *reinterpret_cast<const uint2*>(row);
    u[0] = t.x; u[1] = t.y;
  }
  float x[EPL];
#pragma unroll
  for (int e = 0; e < EPL / 2; ++e) {
    x[2 * e] = __uint_as_float(u[e] << 16);
    x[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
  }
  uint32_t q[EPL / 4];
  const float s = quantize_e4m3_warp<EPL>(x, q);
  uint32_t* dst = reinterpret_cast<uint32_t*>(Wq + v * r + lane * EPL);
#pragma unroll
  for (int w = 0; w < EPL / 4; ++w) dst[w] = q[w];
  if (lane == 0) sw[v] = s;
}

// TMA descriptor of W (2-D: r elements inner, V rows) with 64-element x `rows` boxes, 128-byte swizzle and
// zero fill outside the tensor.
int encode_w(CUtensorMap* m, const void* W, int64_t V, int r, int rows) {
  auto encode = get_encode();
  if (!encode) return WHEAD_ERR_CUDA;
  cuuint64_t gdim[2] = {(cuuint64_t)r, (cuuint64_t)V};
  cuuint64_t gstride[1] = {(cuuint64_t)r * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)rows};
  cuuint32_t estride[2] = {1, 1};
  CUresult cr = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W), gdim, gstride, box, estride,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return cr == CUDA_SUCCESS ? WHEAD_OK : WHEAD_ERR_CUDA;
}

}  // namespace

extern "C" {

int whead_quantize_w_e4m3(const void* W, int64_t V, int32_t r, void* Wq, float* sw, void* stream) {
  if (!W || !Wq || !sw || V < 1) return WHEAD_ERR_INVALID_ARG;
  if (r != 128 && r != 256) return WHEAD_ERR_UNSUPPORTED;
  if (V >= (int64_t)1 << 24) return WHEAD_ERR_UNSUPPORTED;
  if (!aligned16(W) || !aligned16(Wq) || (reinterpret_cast<uintptr_t>(sw) & 3u)) return WHEAD_ERR_INVALID_ARG;
  const unsigned blocks = (unsigned)((V + 7) / 8);  // 8 rows (warps) per block
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t* w = static_cast<const uint16_t*>(W);
  uint8_t* q = static_cast<uint8_t*>(Wq);
  if (r == 256) quantize_w_e4m3_kernel<8><<<blocks, 256, 0, s>>>(w, V, r, q, sw);
  else quantize_w_e4m3_kernel<4><<<blocks, 256, 0, s>>>(w, V, r, q, sw);
  return cudaGetLastError() == cudaSuccess ? WHEAD_OK : WHEAD_ERR_CUDA;
}

const char* whead_strerror(int code) {
  switch (code) {
    case WHEAD_OK: return "ok";
    case WHEAD_ERR_INVALID_ARG: return "invalid argument";
    case WHEAD_ERR_UNSUPPORTED: return "unsupported shape or configuration";
    case WHEAD_ERR_CUDA: return "CUDA call failed";
    case WHEAD_ERR_TIMEOUT: return "a device-side wait ran past its time limit";
    case WHEAD_ERR_NO_COOP: return "grid cannot be co-resident (cooperative launch refused)";
    case WHEAD_ERR_INTERNAL: return "device-side consistency check failed";
    default: return "unknown error";
  }
}

int whead_create(const void* W, const void* E, const whead_params* params, whead_t** out) {
  if (!W || !E || !params || !out) return WHEAD_ERR_INVALID_ARG;
  *out = nullptr;
  const whead_params& p = *params;
  if (p.kind != WHEAD_MARKOV && p.kind != WHEAD_RECURRENT) return WHEAD_ERR_INVALID_ARG;
  if (p.V < 1 || p.max_B < 1 || p.max_B > kMaxB || p.max_gamma < 1 || p.max_gamma > kMaxGamma)
    return WHEAD_ERR_INVALID_ARG;
  if (p.V >= (int64_t)1 << 24) return WHEAD_ERR_UNSUPPORTED;
  if (p.r != 64 && p.r != 128 && p.r != 192 && p.r != 256) return WHEAD_ERR_UNSUPPORTED;
  if (p.kind == WHEAD_RECURRENT && !p.A) return WHEAD_ERR_UNSUPPORTED;
  if (!aligned16(W) || !aligned16(E)) return WHEAD_ERR_INVALID_ARG;
  const bool f8 = (p.flags & WHEAD_FLAG_W_E4M3) != 0u;
  if (f8 && ((p.r != 128 && p.r != 256) || p.max_B > 4)) return WHEAD_ERR_UNSUPPORTED;
  if (p.v_offset < 0 || (p.v_offset & 15) || p.e_rows < 0) return WHEAD_ERR_INVALID_ARG;
  if (p.v_offset + p.V >= (int64_t)1 << 24 || p.e_rows >= (int64_t)1 << 24) return WHEAD_ERR_UNSUPPORTED;
  if (p.e_rows > 0 && p.e_rows < p.v_offset + p.V) return WHEAD_ERR_INVALID_ARG;

  whead_t* h = new (std::nothrow) whead_s();
  if (!h) return WHEAD_ERR_INVALID_ARG;
  h->p = p;
  h->W = static_cast<const uint16_t*>(W);
  h->E = static_cast<const uint16_t*>(E);
  h->f8 = f8;
  h->stream = static_cast<cudaStream_t>(p.stream);
  if (h->p.timeout_us == 0) h->p.timeout_us = 1000000u;
  auto fail = [&](int code) {
    whead_destroy(h);
    return code;
  };
  if (cudaGetDevice(&h->device) != cudaSuccess) return fail(WHEAD_ERR_CUDA);
  if (cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess)
    return fail(WHEAD_ERR_CUDA);
  if (cudaDeviceGetAttribute(&h->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device) != cudaSuccess)
    return fail(WHEAD_ERR_CUDA);
  int coop = 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->device) != cudaSuccess || !coop)
    return fail(WHEAD_ERR_NO_COOP);
  if (cudaDeviceGetAttribute(&h->pageable_access, cudaDevAttrPageableMemoryAccess, h->device) != cudaSuccess)
    return fail(WHEAD_ERR_CUDA);

  h->slots_per_parity = 2 * (int64_t)h->sm_count * kMaxB;

  // placements: walks <= 8 (one n8 half) and, if asked for, walks <= 16
  // measurement modes: nothing on chip (FORCE_STREAM), or caller-chosen caps per tier (PLACEMENT_CAPS)
  int cap_s = INT_MAX, cap_t = INT_MAX, cap_r = INT_MAX;
  const bool force_stream = (p.flags & WHEAD_FLAG_FORCE_STREAM) != 0u;
  const bool capped = (p.flags & WHEAD_FLAG_PLACEMENT_CAPS) != 0u;
  if (force_stream) {
    cap_s = cap_t = cap_r = 0;
  } else if (capped) {
    if (p.cap_smem < 0 || p.cap_tmem < 0 || p.cap_rf < 0) return fail(WHEAD_ERR_INVALID_ARG);
    cap_s = p.cap_smem;
    cap_t = p.cap_tmem;
    cap_r = p.cap_rf;
  }
  const bool fixed = force_stream || capped;
  h->plan[0] = make_plan(p.V, p.r, p.kind, std::min(p.max_B, 8), 1, h->sm_count, h->smem_optin, p.grid, cap_s, cap_t,
                         cap_r, fixed, f8);
  if (!h->plan[0].ok) return fail(WHEAD_ERR_UNSUPPORTED);
  if (p.max_B > 8) {
    h->plan[1] = make_plan(p.V, p.r, p.kind, p.max_B, 2, h->sm_count, h->smem_optin, p.grid, cap_s, cap_t, cap_r,
                           fixed);
    if (!h->plan[1].ok) return fail(WHEAD_ERR_UNSUPPORTED);
  }

  // E4M3 weights: the handle quantizes W once into its own copy (codes and row scales)
  const void* Wt = W;
  int rw = p.r;
  if (f8) {
    if (cudaMalloc(&h->wq, (size_t)p.V * p.r) != cudaSuccess) return fail(WHEAD_ERR_CUDA);
    if (cudaMalloc(&h->sw, (size_t)p.V * 4) != cudaSuccess) return fail(WHEAD_ERR_CUDA);
    const int rc = whead_quantize_w_e4m3(W, p.V, p.r, h->wq, h->sw, h->stream);
    if (rc != WHEAD_OK) return fail(rc);
    Wt = h->wq;
    rw = p.r / 2;  // the codes, described to TMA as pairs: rows of r / 2 16-bit words
  }

  // TMA descriptors of W: 64 x 16 and 64 x 128 boxes of 16-bit words
  if (encode_w(&h->tmap, Wt, p.V, rw, kGroupRows) != WHEAD_OK) return fail(WHEAD_ERR_CUDA);
  if (encode_w(&h->tmap128, Wt, p.V, rw, kGroupRows * kTmaChunkGroups) != WHEAD_OK) return fail(WHEAD_ERR_CUDA);

  // scratch: exchange slots (two call parities), two counters on their own lines, A h slices (two call
  // parities), status word
  const size_t slots_bytes = 2 * (size_t)h->slots_per_parity * 8;
  const size_t cnt_bytes = 256;
  const size_t ah_bytes = 2 * ah_words_per_parity(p.r) * 8;
  const size_t total = slots_bytes + cnt_bytes + ah_bytes + 256;
  if (cudaMalloc(&h->scratch_block, total) != cudaSuccess) return fail(WHEAD_ERR_CUDA);
  if (cudaMemset(h->scratch_block, 0, total) != cudaSuccess) return fail(WHEAD_ERR_CUDA);
  uint8_t* b = static_cast<uint8_t*>(h->scratch_block);
  h->s.slots = reinterpret_cast<unsigned long long*>(b);
  h->s.cnt = reinterpret_cast<unsigned int*>(b + slots_bytes);
  h->s.ah = reinterpret_cast<unsigned long long*>(b + slots_bytes + cnt_bytes);
  h->s.status = reinterpret_cast<int*>(b + slots_bytes + cnt_bytes + ah_bytes);
  *out = h;
  return WHEAD_OK;
}

namespace {
int walk_impl(whead_t* h, const float* base, const float* s0, int32_t B, int32_t gamma, float T, uint64_t seed,
              int64_t t0, int32_t* out_tokens, uint64_t* out_keys, void* out_logits, float* out_state,
              bool base_async = false);
}  // namespace

int whead_walk_keys(whead_t* h, const float* base, const float* s0, int32_t B, int32_t gamma, float T, uint64_t seed,
                    int64_t t0, int32_t* out_tokens, uint64_t* out_keys, void* out_logits, float* out_state) {
  return walk_impl(h, base, s0, B, gamma, T, seed, t0, out_tokens, out_keys, out_logits, out_state);
}

namespace {
int walk_impl(whead_t* h, const float* base, const float* s0, int32_t B, int32_t gamma, float T, uint64_t seed,
              int64_t t0, int32_t* out_tokens, uint64_t* out_keys, void* out_logits, float* out_state,
              bool base_async) {
  if (!h || !base || !s0 || !out_tokens) return WHEAD_ERR_INVALID_ARG;
  if (out_keys && (reinterpret_cast<uintptr_t>(out_keys) & 7u)) return WHEAD_ERR_INVALID_ARG;
  if (B < 1 || B > h->p.max_B || gamma < 1 || gamma > h->p.max_gamma || t0 < 0) return WHEAD_ERR_INVALID_ARG;
  if (!(T >= 0.0f) || T != T || T > 3.0e38f) return WHEAD_ERR_INVALID_ARG;
  if (!aligned16(s0) || (out_state && !aligned16(out_state))) return WHEAD_ERR_INVALID_ARG;
  const int NH = B <= 8 ? 1 : 2;
  const Plan& pl = h->plan[NH - 1];
  if (!pl.ok) return WHEAD_ERR_UNSUPPORTED;

  WalkArgs a;
  std::memset(&a, 0, sizeof(a));
  a.W = h->f8 ? reinterpret_cast<const uint16_t*>(h->wq) : h->W;
  a.sw = h->f8 ? h->sw : nullptr;
  a.rw = h->f8 ? h->p.r / 2 : h->p.r;
  a.E = h->E;
  a.A = h->p.A;
  a.c = h->p.c;
  a.base = base;
  a.s0 = s0;
  a.tokens = out_tokens;
  a.keys = reinterpret_cast<unsigned long long*>(out_keys);
  a.logits = out_logits;
  a.state = out_state;
  const uint32_t par = h->parity & 1u;
  a.slots = h->s.slots + (size_t)par * h->slots_per_parity;
  a.cnt = h->s.cnt + par * 32;
  a.slots_reset = h->s.slots + (size_t)(par ^ 1u) * h->slots_per_parity;
  a.slots_reset_count = (int32_t)h->slots_per_parity;
  a.cnt_reset = h->s.cnt + (par ^ 1u) * 32;
  a.ah = h->s.ah + (size_t)par * ah_words_per_parity(h->p.r);
  a.ah_reset = h->s.ah + (size_t)(par ^ 1u) * ah_words_per_parity(h->p.r);
  a.ah_reset_count = (int32_t)ah_words_per_parity(h->p.r);
  a.status = h->s.status;
  if (h->trace && h->trace_bytes >= (int64_t)pl.G * trace_stride_for(gamma) * 8) {
    a.trace = h->trace;
    a.trace_stride = trace_stride_for(gamma);
  }
  a.V = h->p.V;
  a.v_offset = h->p.v_offset;
  a.t0 = t0;
  a.seed = seed;
  a.timeout_ns = (uint64_t)h->p.timeout_us * 1000ull;
  a.T = T;
  a.r = h->p.r;
  a.B = B;
  a.gamma = gamma;
  a.kind = h->p.kind;
  a.flags = h->p.flags & ~kFlagBaseAsync;
  // base logits behind a slow link: copy each step's rows during the step before, where shared memory allows
  if (base_async && pl.smem_bytes + base_in_bytes(B, pl.ng) <= h->smem_optin) a.flags |= kFlagBaseAsync;
  a.ng = pl.ng;
  a.n_smem = pl.n_smem;
  a.n_tmem = pl.n_tmem;
  a.n_rf = pl.n_rf;
  a.n_stream = pl.n_stream;
  a.tmem_cols = pl.tmem_cols;
  a.smem_w_bytes = pl.smem_w_bytes;
  a.ra = pl.ra;
  a.rf_warp_mask = pl.rf_warp_mask;
  a.ah_warp = pl.ah_warp;
  std::memcpy(a.wl_count, pl.wl_count, sizeof(a.wl_count));
  std::memcpy(a.wl, pl.wl, sizeof(a.wl));
  const int rc = launch(h, pl, a, NH);
  if (rc == WHEAD_OK) h->parity ^= 1u;
  return rc;
}
}  // namespace

int whead_walk_ex(whead_t* h, const float* base, const float* s0, int32_t B, int32_t gamma, float T, uint64_t seed,
                  int64_t t0, int32_t* out_tokens, void* out_logits, float* out_state) {
  return whead_walk_keys(h, base, s0, B, gamma, T, seed, t0, out_tokens, nullptr, out_logits, out_state);
}

int whead_walk(whead_t* h, const float* base, const float* u0, int32_t B, int32_t gamma, float T, uint64_t seed,
               int32_t* out_tokens, void* out_logits) {
  return whead_walk_ex(h, base, u0, B, gamma, T, seed, 0, out_tokens, out_logits, nullptr);
}

int whead_advance(whead_t* h, const int32_t* x, const float* s, float* s_next, int32_t B) {
  if (!h || !x || !s || !s_next) return WHEAD_ERR_INVALID_ARG;
  if (B < 1 || B > h->p.max_B) return WHEAD_ERR_INVALID_ARG;
  const int64_t e_rows = h->p.e_rows > 0 ? h->p.e_rows : h->p.v_offset + h->p.V;
  const int warps = B * h->p.r;
  advance_kernel<<<(warps + 7) / 8, 256, 0, h->stream>>>(h->p.kind, h->E, h->p.A, h->p.c, x, s, s_next, B, h->p.r,
                                                       e_rows, h->s.status);
  return cudaGetLastError() == cudaSuccess ? WHEAD_OK : WHEAD_ERR_CUDA;
}

namespace {
// A pointer this GPU can reach the caller's memory through, or nullptr: memory of this device, managed
// memory, host memory pinned and mapped by CUDA, or any host memory where the GPU walks the host's page
// tables (as on Grace over NVLink-C2C).
void* device_view(const whead_t* h, const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice: return at.device == h->device ? const_cast<void*>(p) : nullptr;
    case cudaMemoryTypeManaged: return const_cast<void*>(p);
    case cudaMemoryTypeHost: return at.devicePointer;
    default: return h->pageable_access ? const_cast<void*>(p) : nullptr;
  }
}
}  // namespace

int whead_walk_host(whead_t* h, const float* base_host, const float* u0_host, int32_t B, int32_t gamma, float T,
                    uint64_t seed, int32_t* out_tokens_host, void* out_logits_host) {
  if (!h || !base_host || !u0_host || !out_tokens_host) return WHEAD_ERR_INVALID_ARG;
  if (B < 1 || B > h->p.max_B || gamma < 1 || gamma > h->p.max_gamma) return WHEAD_ERR_INVALID_ARG;
  const size_t nbase = (size_t)B * gamma * h->p.V;
  const size_t logit_elem = (h->p.flags & WHEAD_FLAG_LOGITS_F32) ? 4 : 2;
  if (!h->d_u0) {
    if (cudaMalloc(&h->d_u0, (size_t)h->p.max_B * h->p.r * 4) != cudaSuccess) return WHEAD_ERR_CUDA;
    if (cudaMalloc(&h->d_tok, (size_t)h->p.max_B * h->p.max_gamma * 4) != cudaSuccess) return WHEAD_ERR_CUDA;
    if (cudaMallocHost(&h->h_status, sizeof(int)) != cudaSuccess) return WHEAD_ERR_CUDA;
  }
  if (out_logits_host && !h->d_logits) {
    const size_t cap = (size_t)h->p.max_B * h->p.max_gamma * h->p.V;
    if (cudaMalloc(&h->d_logits, cap * logit_elem) != cudaSuccess) return WHEAD_ERR_CUDA;
  }
  // The walk reads each step's base logits where the caller keeps them when the GPU can address that memory,
  // copying step t + 1's rows into shared memory asynchronously during step t, which hides the host link's
  // latency; it reads u0 and writes the tokens in place on the same condition. Whatever it cannot reach is
  // copied through handle-owned device buffers.
  const bool stage = (h->p.flags & WHEAD_FLAG_HOST_STAGE) != 0u;
  const float* base = stage ? nullptr : static_cast<const float*>(device_view(h, base_host));
  const bool in_place = base != nullptr;
  if (!base) {
    if (!h->d_base) {
      const size_t cap = (size_t)h->p.max_B * h->p.max_gamma * h->p.V;
      if (cudaMalloc(&h->d_base, cap * 4) != cudaSuccess) return WHEAD_ERR_CUDA;
    }
    if (cudaMemcpyAsync(h->d_base, base_host, nbase * 4, cudaMemcpyDefault, h->stream) != cudaSuccess)
      return WHEAD_ERR_CUDA;
    base = h->d_base;
  }
  const float* u0 = stage ? nullptr : static_cast<const float*>(device_view(h, u0_host));
  if (!u0 || !aligned16(u0)) {
    if (cudaMemcpyAsync(h->d_u0, u0_host, (size_t)B * h->p.r * 4, cudaMemcpyDefault, h->stream) != cudaSuccess)
      return WHEAD_ERR_CUDA;
    u0 = h->d_u0;
  }
  int32_t* tok = stage ? nullptr : static_cast<int32_t*>(device_view(h, out_tokens_host));
  if (!tok) tok = h->d_tok;
  const int rc = walk_impl(h, base, u0, B, gamma, T, seed, 0, tok, nullptr, out_logits_host ? h->d_logits : nullptr,
                           nullptr, in_place);
  if (rc != WHEAD_OK) return rc;
  if (tok == h->d_tok &&
      cudaMemcpyAsync(out_tokens_host, h->d_tok, (size_t)B * gamma * 4, cudaMemcpyDefault, h->stream) != cudaSuccess)
    return WHEAD_ERR_CUDA;
  if (out_logits_host &&
      cudaMemcpyAsync(out_logits_host, h->d_logits, nbase * logit_elem, cudaMemcpyDefault, h->stream) != cudaSuccess)
    return WHEAD_ERR_CUDA;
  if (cudaMemcpyAsync(h->h_status, h->s.status, sizeof(int), cudaMemcpyDeviceToHost, h->stream) != cudaSuccess)
    return WHEAD_ERR_CUDA;
  if (cudaStreamSynchronize(h->stream) != cudaSuccess) return WHEAD_ERR_CUDA;
  const int st = *h->h_status;
  if (st != 0) {  // report the device-side error once, as whead_status does
    if (cudaMemsetAsync(h->s.status, 0, sizeof(int), h->stream) != cudaSuccess) return WHEAD_ERR_CUDA;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return WHEAD_ERR_CUDA;
  }
  return st;
}

int whead_set_trace(whead_t* h, void* trace, int64_t bytes) {
  if (!h || bytes < 0 || (trace && (reinterpret_cast<uintptr_t>(trace) & 7u))) return WHEAD_ERR_INVALID_ARG;
  h->trace = static_cast<unsigned long long*>(trace);
  h->trace_bytes = trace ? bytes : 0;
  return WHEAD_OK;
}

int whead_status(whead_t* h) {
  if (!h) return WHEAD_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(h->stream) != cudaSuccess) return WHEAD_ERR_CUDA;
  int st = 0;
  if (cudaMemcpy(&st, h->s.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return WHEAD_ERR_CUDA;
  if (st != 0) {
    const int zero = 0;
    if (cudaMemcpy(h->s.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return WHEAD_ERR_CUDA;
  }
  return st;
}

int whead_plan_info(const whead_t* h, int32_t B, whead_plan* out) {
  if (!h || !out || B < 1 || B > h->p.max_B) return WHEAD_ERR_INVALID_ARG;
  const Plan& pl = h->plan[B <= 8 ? 0 : 1];
  if (!pl.ok) return WHEAD_ERR_UNSUPPORTED;
  out->grid = pl.G;
  out->threads = kThreads;
  out->groups_per_cta = pl.ng;
  out->smem_groups = pl.n_smem;
  out->tmem_groups = pl.n_tmem;
  out->rf_groups = pl.n_rf;
  out->stream_groups = pl.n_stream;
  out->smem_bytes = pl.smem_bytes;
  out->tmem_cols = (int32_t)pl.tmem_cols;
  out->sm_count = h->sm_count;
  return WHEAD_OK;
}

int whead_plan_query(int64_t V, int32_t r, int32_t kind, int32_t max_B, int32_t B, uint32_t flags, int32_t sm_count,
                     int32_t smem_optin, whead_plan* out, uint32_t* work_lists, uint32_t* rf_warp_mask,
                     int32_t* ah_warp) {
  if (!out || (kind != WHEAD_MARKOV && kind != WHEAD_RECURRENT)) return WHEAD_ERR_INVALID_ARG;
  if (V < 1 || max_B < 1 || max_B > kMaxB || B < 1 || B > max_B || sm_count < 1 || smem_optin < 1)
    return WHEAD_ERR_INVALID_ARG;
  if (V >= (int64_t)1 << 24) return WHEAD_ERR_UNSUPPORTED;
  if (r != 64 && r != 128 && r != 192 && r != 256) return WHEAD_ERR_UNSUPPORTED;
  const bool f8 = (flags & WHEAD_FLAG_W_E4M3) != 0u;
  if (f8 && ((r != 128 && r != 256) || max_B > 4)) return WHEAD_ERR_UNSUPPORTED;
  // the same two plans whead_create makes: up to 8 walks (one n8 half), and up to 16
  const Plan pl = B <= 8 ? make_plan(V, r, kind, std::min(max_B, 8), 1, sm_count, smem_optin, 0, INT_MAX, INT_MAX,
                                     INT_MAX, false, f8)
                         : make_plan(V, r, kind, max_B, 2, sm_count, smem_optin, 0);
  if (!pl.ok) return WHEAD_ERR_UNSUPPORTED;
  out->grid = pl.G;
  out->threads = kThreads;
  out->groups_per_cta = pl.ng;
  out->smem_groups = pl.n_smem;
  out->tmem_groups = pl.n_tmem;
  out->rf_groups = pl.n_rf;
  out->stream_groups = pl.n_stream;
  out->smem_bytes = pl.smem_bytes;
  out->tmem_cols = (int32_t)pl.tmem_cols;
  out->sm_count = sm_count;
  if (work_lists) {
    for (int w = 0; w < kWarps; ++w) {
      uint32_t* row = work_lists + (size_t)w * (1 + kMaxWarpGroups);
      row[0] = (uint32_t)pl.wl_count[w];
      for (int e = 0; e < kMaxWarpGroups; ++e) row[1 + e] = e < pl.wl_count[w] ? pl.wl[w][e] : 0u;
    }
  }
  if (rf_warp_mask) *rf_warp_mask = pl.rf_warp_mask;
  if (ah_warp) *ah_warp = pl.ah_warp;
  return WHEAD_OK;
}

int whead_destroy(whead_t* h) {
  if (!h) return WHEAD_ERR_INVALID_ARG;
  int rc = WHEAD_OK;
  if (h->scratch_block || h->d_base) {
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) rc = WHEAD_ERR_CUDA;
  }
  if (h->scratch_block) cudaFree(h->scratch_block);
  if (h->wq) cudaFree(h->wq);
  if (h->sw) cudaFree(h->sw);
  if (h->d_base) cudaFree(h->d_base);
  if (h->h_status) cudaFreeHost(h->h_status);
  if (h->d_u0) cudaFree(h->d_u0);
  if (h->d_tok) cudaFree(h->d_tok);
  if (h->d_logits) cudaFree(h->d_logits);
  delete h;
  return rc;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// Entry point without allocation: the scratch lives in one file-scope device array.
// ------------------------------------------------------------------------------------------------
namespace {

// Layout of the array: [slots: 2 step parities x 16 walks x up to 256 CTAs, 64 KB][counter 128 B][status 128 B]
// [tagged A h slices: 2 step parities x B x r words, up to 64 KB]. Slots, counter, status and the slices of
// the call are cleared by the host before every call.
constexpr int kNaMaxGrid = kMaxGrid;
constexpr size_t kNaSlots = 2 * (size_t)kNaMaxGrid * kMaxB * 8;
constexpr size_t kNaCntOff = kNaSlots;
constexpr size_t kNaStatusOff = kNaCntOff + 128;
constexpr size_t kNaAhOff = kNaStatusOff + 128;
static_assert(kNaAhOff + 2 * (size_t)kMaxB * 256 * 8 <= WHEAD_NOALLOC_SCRATCH_BYTES, "scratch array too small");

static __device__ __align__(256) unsigned char g_noalloc_scratch[WHEAD_NOALLOC_SCRATCH_BYTES];

constexpr int kNaMaxDevices = 64;
struct NaDevice {
  void* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int sm_count = 0, smem_optin = 0, coop = 0;
  bool ready = false;
};
NaDevice g_na_devices[kNaMaxDevices];

// Once per device, with that device current: the array's device address and the device limits.
int noalloc_setup(int dev, NaDevice** out) {
  if (dev < 0 || dev >= kNaMaxDevices) return WHEAD_ERR_UNSUPPORTED;
  NaDevice& d = g_na_devices[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return WHEAD_ERR_CUDA;
    }
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
      return WHEAD_ERR_CUDA;
    d.scratch = p;
    d.ready = true;
  }
  *out = &d;
  return WHEAD_OK;
}

int noalloc_launch(int r, int NH, const CUtensorMap& tmap, const CUtensorMap& tmap128, cudaStream_t stream,
                   int smem_optin, const Plan& pl, const WalkArgs& a) {
  const WalkLaunch l{&tmap, &tmap128, stream, smem_optin, pl.G, pl.smem_bytes, r, NH, false};
  return a.kind == WHEAD_RECURRENT ? launch_walk_resident_recurrent(l, a) : launch_walk_resident_markov(l, a);
}

}  // namespace

extern "C" int whead_walk_noalloc(const void* W, const void* E, const whead_params* params, const float* base,
                                  const float* u0, int32_t B, int32_t gamma, float T, uint64_t seed,
                                  int32_t* out_tokens, void* out_logits, int32_t* out_status) {
  if (!W || !E || !params || !base || !u0 || !out_tokens) return WHEAD_ERR_INVALID_ARG;
  const whead_params& p = *params;
  if (p.kind != WHEAD_MARKOV && p.kind != WHEAD_RECURRENT) return WHEAD_ERR_INVALID_ARG;
  if (p.V < 1 || B < 1 || gamma < 1) return WHEAD_ERR_INVALID_ARG;
  if (B > kMaxB || gamma > kMaxGamma) return WHEAD_ERR_UNSUPPORTED;  // beyond the scratch array's sizes
  if (p.V >= (int64_t)1 << 24) return WHEAD_ERR_UNSUPPORTED;
  if (p.r != 64 && p.r != 128 && p.r != 192 && p.r != 256) return WHEAD_ERR_UNSUPPORTED;
  if (p.kind == WHEAD_RECURRENT && !p.A) return WHEAD_ERR_UNSUPPORTED;
  // E4M3 needs the handle's quantized copy of W; the measurement and staging modes need a handle's plans
  if (p.flags & (WHEAD_FLAG_W_E4M3 | WHEAD_FLAG_FORCE_STREAM | WHEAD_FLAG_PLACEMENT_CAPS | WHEAD_FLAG_HOST_STAGE))
    return WHEAD_ERR_UNSUPPORTED;
  if (p.v_offset < 0 || (p.v_offset & 15)) return WHEAD_ERR_INVALID_ARG;
  if (p.v_offset + p.V >= (int64_t)1 << 24) return WHEAD_ERR_UNSUPPORTED;
  if (!(T >= 0.0f) || T > 3.0e38f) return WHEAD_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(E) || !aligned16(u0)) return WHEAD_ERR_INVALID_ARG;
  const size_t need = kNaAhOff + 2 * (size_t)B * p.r * 8;
  if (need > WHEAD_NOALLOC_SCRATCH_BYTES) return WHEAD_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return WHEAD_ERR_CUDA;
  NaDevice* nd = nullptr;
  int rc = noalloc_setup(dev, &nd);
  if (rc != WHEAD_OK) return rc;
  if (!nd->coop) return WHEAD_ERR_NO_COOP;

  const int NH = B <= 8 ? 1 : 2;
  const Plan pl = make_plan(p.V, p.r, p.kind, B, NH, nd->sm_count, nd->smem_optin, 0);
  if (!pl.ok) return WHEAD_ERR_UNSUPPORTED;
  static_assert(kMaxGrid <= kNaMaxGrid, "the planner caps the grid at the array's slots per step");

  CUtensorMap tmap, tmap128;
  if (encode_w(&tmap, W, p.V, p.r, kGroupRows) != WHEAD_OK) return WHEAD_ERR_CUDA;
  if (encode_w(&tmap128, W, p.V, p.r, kGroupRows * kTmaChunkGroups) != WHEAD_OK) return WHEAD_ERR_CUDA;

  cudaStream_t stream = static_cast<cudaStream_t>(p.stream);
  uint8_t* sc = static_cast<uint8_t*>(nd->scratch);
  if (cudaMemsetAsync(sc, 0, 2 * (size_t)pl.G * B * 8, stream) != cudaSuccess) return WHEAD_ERR_CUDA;
  if (cudaMemsetAsync(sc + kNaCntOff, 0, 256, stream) != cudaSuccess) return WHEAD_ERR_CUDA;
  if (p.kind == WHEAD_RECURRENT && cudaMemsetAsync(sc + kNaAhOff, 0, 2 * (size_t)B * p.r * 8, stream) != cudaSuccess)
    return WHEAD_ERR_CUDA;
  if (out_status && cudaMemsetAsync(out_status, 0, sizeof(int32_t), stream) != cudaSuccess) return WHEAD_ERR_CUDA;

  WalkArgs a;
  std::memset(&a, 0, sizeof(a));
  a.W = static_cast<const uint16_t*>(W);
  a.sw = nullptr;
  a.rw = p.r;
  a.E = static_cast<const uint16_t*>(E);
  a.A = p.A;
  a.c = p.c;
  a.base = base;
  a.s0 = u0;
  a.tokens = out_tokens;
  a.logits = out_logits;
  a.state = nullptr;
  a.slots = reinterpret_cast<unsigned long long*>(sc);
  a.cnt = reinterpret_cast<unsigned int*>(sc + kNaCntOff);
  a.slots_reset = nullptr;  // cleared above by the host
  a.cnt_reset = nullptr;
  a.ah = reinterpret_cast<unsigned long long*>(sc + kNaAhOff);
  a.ah_reset = nullptr;  // cleared above by the host
  a.status = out_status ? reinterpret_cast<int*>(out_status) : reinterpret_cast<int*>(sc + kNaStatusOff);
  a.V = p.V;
  a.v_offset = p.v_offset;
  a.t0 = 0;
  a.seed = seed;
  a.timeout_ns = (uint64_t)(p.timeout_us ? p.timeout_us : 1000000u) * 1000ull;
  a.T = T;
  a.r = p.r;
  a.B = B;
  a.gamma = gamma;
  a.kind = p.kind;
  a.flags = p.flags & ~kFlagBaseAsync;  // the library-internal launch bit is never the caller's
  a.ng = pl.ng;
  a.n_smem = pl.n_smem;
  a.n_tmem = pl.n_tmem;
  a.n_rf = pl.n_rf;
  a.n_stream = pl.n_stream;
  a.tmem_cols = pl.tmem_cols;
  a.smem_w_bytes = pl.smem_w_bytes;
  a.ra = pl.ra;
  a.rf_warp_mask = pl.rf_warp_mask;
  a.ah_warp = pl.ah_warp;
  std::memcpy(a.wl_count, pl.wl_count, sizeof(a.wl_count));
  std::memcpy(a.wl, pl.wl, sizeof(a.wl));
  return noalloc_launch(p.r, NH, tmap, tmap128, stream, nd->smem_optin, pl, a);
}
