// onchip_probe.cu — measures the per-SM figures the walk's on-chip roofline is expressed in.
//
// Built as a separate library (libwhead_probe.so) for the benchmark; the walk library does not use it.
//   whead_probe_onchip(out[6]):
//     out[0] shared-memory read bandwidth, bytes per SM clock (ld.shared.v4, 384 threads, 192 KB resident)
//     out[1] tensor-memory read bandwidth, bytes per SM clock (two tcgen05.ld.32x32b.x64 in flight per wait,
//            384 threads, 512 columns)
//     out[2] SM clocks per mma.sync.m16n8k16 bf16 -> fp32 per SM (independent accumulators, 384 threads)
//     out[3] SM clocks per grid-wide arrival + wait over all SMs (relaxed counter; cooperative launch)
//     out[4] SM clocks per tcgen05.mma.cta_group::1.kind::f16 of shape M128 N16 K16 (A and B in shared memory,
//            128-byte swizzle, D in tensor memory), one issuing thread
//     out[5] the same with four issuing threads (one per warp, separate accumulators)
//     out[6] SM clocks for 256 of those M128 N16 K16 instructions from one thread while 11 warps stay idle
//     out[7] SM clocks for 11 warps running 800 mma.sync.m16n8k16 each while that thread stays idle
//     out[8] SM clocks for the 11 warps' mma.sync when the thread issues its tcgen05.mma at the same time
// out[4] and out[5] say how fast the fifth-generation tensor core consumes a thin (N <= 16) operand: W bytes per
// clock = 4096 / out[5], against 256 B per clock for mma.sync.m16n8k16 at out[2] = 2. out[6..8] say whether the
// two can share the projection: if they ran side by side, out[8] would stay near out[7].
// Every wait is bounded; every access stays inside its buffer. Returns 0, or a negative CUDA error.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

namespace {

constexpr int kThreads = 384;

__global__ void __launch_bounds__(kThreads, 1) smem_bw(uint32_t* out, long long* cyc, int iters, int bytes) {
  extern __shared__ __align__(16) uint8_t sm[];
  uint32_t* s = reinterpret_cast<uint32_t*>(sm);
  for (int i = threadIdx.x; i < bytes / 4; i += blockDim.x) s[i] = i * 2654435761u;
  __syncthreads();
  uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
  const int n16 = bytes / 16;
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll 4
    for (int i = threadIdx.x; i < n16; i += blockDim.x) {
      const uint4 v = reinterpret_cast<const uint4*>(sm)[i];
      a0 ^= v.x; a1 ^= v.y; a2 ^= v.z; a3 ^= v.w;
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  out[blockIdx.x * blockDim.x + threadIdx.x] = a0 ^ a1 ^ a2 ^ a3;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// 64 columns of this warp's lane quadrant in one load (32 lanes x 64 x 4 B = 8 KB per warp)
#define WH_TMEM_X64_OUT(r)                                                                                          \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),      \
      "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),       \
      "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),      \
      "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]),      \
      "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]),      \
      "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),      \
      "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]),      \
      "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
#define WH_TMEM_X64_ASM                                                                                             \
  "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"  \
  "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47," \
  "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"

// Tensor-memory read bandwidth with loads kept in flight: each warp issues two 64-column loads (16 KB) and waits
// once, sweeping all 512 columns of its lane quadrant (the three warps of a quadrant each read all of them).
__global__ void __launch_bounds__(kThreads, 1) tmem_bw(uint32_t* out, long long* cyc, int iters) {
  __shared__ uint32_t taddr_s;
  const int warp = threadIdx.x >> 5;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
        (uint32_t)__cvta_generic_to_shared(&taddr_s)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t taddr = taddr_s;
  const int quad = warp & 3;
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  uint32_t acc = 0;
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
    for (int col = 0; col < 512; col += 128) {
      uint32_t r0[64], r1[64];
      asm volatile(WH_TMEM_X64_ASM : WH_TMEM_X64_OUT(r0) : "r"(taddr + lane_base + (uint32_t)col));
      asm volatile(WH_TMEM_X64_ASM : WH_TMEM_X64_OUT(r1) : "r"(taddr + lane_base + (uint32_t)(col + 64)));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
      for (int j = 0; j < 64; ++j) acc ^= r0[j] ^ r1[j];
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  const long long t1 = clock64();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(taddr));
  out[blockIdx.x * blockDim.x + threadIdx.x] = acc;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}
#undef WH_TMEM_X64_ASM
#undef WH_TMEM_X64_OUT

__global__ void __launch_bounds__(kThreads, 1) mma_rate(float* out, long long* cyc, int iters) {
  const uint32_t a0 = threadIdx.x, a1 = threadIdx.x * 3u, a2 = threadIdx.x * 5u, a3 = threadIdx.x * 7u;
  const uint32_t b0 = 0x3f803f80u, b1 = 0x3f803f80u;
  float c[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.f;
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
          : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

__global__ void __launch_bounds__(kThreads, 1) grid_exchange(unsigned int* counter, int* status, long long* cyc,
                                                             int iters) {
  const unsigned int G = gridDim.x;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
    __syncthreads();
    if (threadIdx.x == 0) {
      asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
      const unsigned int target = (unsigned int)(it + 1) * G;
      uint32_t spins = 0;
      while (true) {
        unsigned int v;
        asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
        if (v >= target) break;
        if (++spins > 4000000u) {
          atomicExch(status, 1);
          break;
        }
      }
    }
    __syncthreads();
  }
  const long long t1 = clock64();
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

// --- tcgen05.mma issue rate at a thin N ---
constexpr int kUmmaABytes = 128 * 256 * 2;  // one 128 x 256 bf16 tile, [k/64][128 rows][128 B], 128-byte swizzle
constexpr int kUmmaBBytes = 16 * 256 * 2;   // 16 x 256 bf16, [k/64][16 rows][128 B]
constexpr int kUmmaSmem = kUmmaABytes + kUmmaBBytes + 1024 + 64;

__device__ __forceinline__ uint64_t umma_sdesc(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1u << 16) | ((uint64_t)(1024u >> 4) << 32) |
         ((uint64_t)1u << 46) | ((uint64_t)2u << 61);
}

// NW threads (lane 0 of warps 0..NW-1) each issue 2 tiles x 16 K-steps of M128 N16 K16 into their own columns,
// commit to their own mbarrier and wait (bounded by 100 ms of global time). cyc[block] = issuer 0's median.
template <int NW>
__global__ void __launch_bounds__(128, 1) umma_rate(long long* cyc, int* status, int reps) {
  extern __shared__ uint8_t umma_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(umma_smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + kUmmaABytes + kUmmaBBytes);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(mbar + 4);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  for (int i = tid; i < (kUmmaABytes + kUmmaBBytes) / 16; i += blockDim.x) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(s_tmem)),
                 "r"(256) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid < 4) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"((uint32_t)__cvta_generic_to_shared(mbar + tid)) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *s_tmem;
  __shared__ long long s_med[16];
  if (warp < NW && lane == 0) {
    // instruction descriptor: D f32, A and B bf16, both K-major, N = 16, M = 128
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
    const uint32_t a0 = (uint32_t)__cvta_generic_to_shared(sm), b0 = a0 + kUmmaABytes;
    const uint32_t mb = (uint32_t)__cvta_generic_to_shared(mbar + warp);
    for (int rep = 0; rep < reps && rep < 16; ++rep) {
      const long long t0 = clock64();
#pragma unroll 1
      for (int d = 0; d < 2; ++d) {
        const uint32_t dcol = tmem + (uint32_t)((warp * 2 + d) * 16);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint64_t ad = umma_sdesc(a0 + (uint32_t)((kk / 4) * 128 * 128 + (kk % 4) * 32));
          const uint64_t bd = umma_sdesc(b0 + (uint32_t)((kk / 4) * 16 * 128 + (kk % 4) * 32));
          asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                       " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                       ::"r"(dcol), "l"(ad), "l"(bd), "r"(idesc), "r"(kk > 0 ? 1u : 0u) : "memory");
        }
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mb) : "memory");
      bool ok = false;
      uint64_t ts, tn;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(ts));
      tn = ts;
      while (!ok && tn - ts < 100000000ull) {
        uint32_t r;
        asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(r) : "r"(mb), "r"((uint32_t)(rep & 1)) : "memory");
        ok = r != 0;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tn));
      }
      if (warp == 0) s_med[rep] = clock64() - t0;
      if (!ok) {
        atomicExch(status, 1);
        break;
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (tid == 0) {
    // median of repetitions 2.. (the first two warm up)
    long long v[16];
    const int n = (reps < 16 ? reps : 16) - 2;
    for (int i = 0; i < n; ++i) v[i] = s_med[i + 2];
    for (int i = 1; i < n; ++i)
      for (int j = i; j > 0 && v[j - 1] > v[j]; --j) { const long long x = v[j]; v[j] = v[j - 1]; v[j - 1] = x; }
    cyc[blockIdx.x] = v[n / 2];
  }
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256) : "memory");
}

// tcgen05.mma beside mma.sync. mode 0: warp 11's lane 0 issues `tiles` x 16 M128 N16 K16 (A and B in shared
// memory as above, one accumulator) and waits for them (bounded by 100 ms); mode 1: warps 0-10 run `iters` x 8
// independent mma.sync; mode 2: both at once. cyc[2 b] = the tcgen05 issuer's clocks, cyc[2 b + 1] = the slowest
// mma.sync warp's.
__global__ void __launch_bounds__(kThreads, 1) umma_beside_mma(long long* cyc, int* status, float* sink, int mode,
                                                               int tiles, int iters) {
  extern __shared__ uint8_t umma_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(umma_smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + kUmmaABytes + kUmmaBBytes);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(mbar + 2);
  __shared__ long long s_t[kThreads / 32];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  for (int i = tid; i < (kUmmaABytes + kUmmaBBytes) / 16; i += blockDim.x) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(s_tmem)),
                 "r"(32) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"((uint32_t)__cvta_generic_to_shared(mbar)) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *s_tmem;
  const long long t0 = clock64();
  long long t = 0;
  if (warp == kThreads / 32 - 1) {
    if (lane == 0 && mode != 1) {
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
      const uint32_t a0 = (uint32_t)__cvta_generic_to_shared(sm), b0 = a0 + kUmmaABytes;
      const uint32_t mb = (uint32_t)__cvta_generic_to_shared(mbar);
      for (int tile = 0; tile < tiles; ++tile) {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint64_t ad = umma_sdesc(a0 + (uint32_t)((kk / 4) * 128 * 128 + (kk % 4) * 32));
          const uint64_t bd = umma_sdesc(b0 + (uint32_t)((kk / 4) * 16 * 128 + (kk % 4) * 32));
          asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                       " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                       ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc), "r"(kk > 0 ? 1u : 0u) : "memory");
        }
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mb) : "memory");
      bool ok = false;
      uint64_t ts, tn;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(ts));
      tn = ts;
      while (!ok && tn - ts < 100000000ull) {
        uint32_t r;
        asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n selp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(r) : "r"(mb) : "memory");
        ok = r != 0;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(tn));
      }
      t = clock64() - t0;
      if (!ok) atomicExch(status, 1);
    }
  } else if (mode != 0) {
    const uint32_t a0 = tid, a1 = tid * 3u, a2 = tid * 5u, a3 = tid * 7u;
    const uint32_t b0 = 0x3f803f80u, b1 = 0x3f803f80u;
    float c[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) sum += c[j][0] + c[j][1] + c[j][2] + c[j][3];
    sink[blockIdx.x * blockDim.x + tid] = sum;
    t = clock64() - t0;
  }
  if (lane == 0) s_t[warp] = t;
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (tid == 0) {
    long long mx = 0;
    for (int w = 0; w < kThreads / 32 - 1; ++w) mx = s_t[w] > mx ? s_t[w] : mx;
    cyc[2 * blockIdx.x] = s_t[kThreads / 32 - 1];
    cyc[2 * blockIdx.x + 1] = mx;
  }
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(32) : "memory");
}

double median_cycles(const long long* d_cyc, int n) {
  std::vector<long long> h(n);
  if (cudaMemcpy(h.data(), d_cyc, n * sizeof(long long), cudaMemcpyDeviceToHost) != cudaSuccess) return -1.0;
  std::sort(h.begin(), h.end());
  return (double)h[n / 2];
}

}  // namespace

extern "C" int whead_probe_onchip(double* out) {
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  uint32_t* d_out = nullptr;
  long long* d_cyc = nullptr;
  unsigned int* d_cnt = nullptr;
  int* d_status = nullptr;
  int rc = 0;
  const int smem_bytes = 192 * 1024;
  do {
    if (cudaMalloc(&d_out, (size_t)nsm * kThreads * 4) != cudaSuccess) { rc = -2; break; }
    if (cudaMalloc(&d_cyc, (size_t)nsm * 2 * 8) != cudaSuccess) { rc = -2; break; }
    if (cudaMalloc(&d_cnt, 256) != cudaSuccess) { rc = -2; break; }
    if (cudaMalloc(&d_status, 4) != cudaSuccess) { rc = -2; break; }
    if (cudaFuncSetAttribute(smem_bw, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess) { rc = -3; break; }
    if (cudaFuncSetAttribute(tmem_bw, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024) != cudaSuccess) { rc = -3; break; }
    const int it_smem = 200;
    smem_bw<<<nsm, kThreads, smem_bytes>>>(d_out, d_cyc, 2, smem_bytes);
    smem_bw<<<nsm, kThreads, smem_bytes>>>(d_out, d_cyc, it_smem, smem_bytes);
    if (cudaDeviceSynchronize() != cudaSuccess) { rc = -4; break; }
    out[0] = (double)smem_bytes * it_smem / median_cycles(d_cyc, nsm);
    // 160 KB of dynamic shared memory keeps one CTA per SM, so every CTA owns all 512 columns
    const int it_tmem = 200;
    tmem_bw<<<nsm, kThreads, 160 * 1024>>>(d_out, d_cyc, 2);
    tmem_bw<<<nsm, kThreads, 160 * 1024>>>(d_out, d_cyc, it_tmem);
    if (cudaDeviceSynchronize() != cudaSuccess) { rc = -4; break; }
    out[1] = (double)it_tmem * (kThreads / 128) * 512 * 128 * 4 / median_cycles(d_cyc, nsm);
    const int it_mma = 2000;
    mma_rate<<<nsm, kThreads>>>(reinterpret_cast<float*>(d_out), d_cyc, 10);
    mma_rate<<<nsm, kThreads>>>(reinterpret_cast<float*>(d_out), d_cyc, it_mma);
    if (cudaDeviceSynchronize() != cudaSuccess) { rc = -4; break; }
    out[2] = median_cycles(d_cyc, nsm) / ((double)it_mma * 8 * (kThreads / 32));
    int iters = 1000;
    if (cudaMemset(d_cnt, 0, 256) != cudaSuccess || cudaMemset(d_status, 0, 4) != cudaSuccess) { rc = -4; break; }
    void* args[] = {&d_cnt, &d_status, &d_cyc, &iters};
    if (cudaLaunchCooperativeKernel((const void*)grid_exchange, nsm, kThreads, args, 0, 0) != cudaSuccess) { rc = -5; break; }
    if (cudaDeviceSynchronize() != cudaSuccess) { rc = -4; break; }
    int st = 0;
    cudaMemcpy(&st, d_status, 4, cudaMemcpyDeviceToHost);
    out[3] = st ? -1.0 : median_cycles(d_cyc, nsm) / iters;
    // 120 KB of dynamic shared memory keeps one CTA per SM (the kernel uses the first 74 KB)
    const int umma_smem = 120 * 1024;
    static_assert(kUmmaSmem <= 120 * 1024, "umma probe layout");
    if (cudaFuncSetAttribute(umma_rate<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, umma_smem) != cudaSuccess ||
        cudaFuncSetAttribute(umma_rate<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, umma_smem) != cudaSuccess) { rc = -3; break; }
    if (cudaMemset(d_status, 0, 4) != cudaSuccess) { rc = -4; break; }
    umma_rate<1><<<nsm, 128, umma_smem>>>(d_cyc, d_status, 12);
    if (cudaDeviceSynchronize() != cudaSuccess) { rc = -4; break; }
    out[4] = median_cycles(d_cyc, nsm) / 32.0;
    umma_rate<4><<<nsm, 128, umma_smem>>>(d_cyc, d_status, 12);
    if (cudaDeviceSynchronize() != cudaSuccess) { rc = -4; break; }
    out[5] = median_cycles(d_cyc, nsm) / 128.0;
    cudaMemcpy(&st, d_status, 4, cudaMemcpyDeviceToHost);
    if (st) out[4] = out[5] = -1.0;
    // tcgen05.mma beside mma.sync: (tcgen05 alone, mma.sync alone, mma.sync with tcgen05 at the same time)
    if (cudaFuncSetAttribute(umma_beside_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, umma_smem) != cudaSuccess) { rc = -3; break; }
    if (cudaMemset(d_status, 0, 4) != cudaSuccess) { rc = -4; break; }
    float* d_sink = reinterpret_cast<float*>(d_out);  // nsm x kThreads floats
    double med[3] = {0, 0, 0};
    for (int mode = 0; mode < 3; ++mode) {
      umma_beside_mma<<<nsm, kThreads, umma_smem>>>(d_cyc, d_status, d_sink, mode, 16, 100);  // warm-up
      umma_beside_mma<<<nsm, kThreads, umma_smem>>>(d_cyc, d_status, d_sink, mode, 16, 100);
      if (cudaDeviceSynchronize() != cudaSuccess) { rc = -4; break; }
      std::vector<long long> h(2 * nsm), a(nsm);
      if (cudaMemcpy(h.data(), d_cyc, 2 * nsm * sizeof(long long), cudaMemcpyDeviceToHost) != cudaSuccess) { rc = -4; break; }
      for (int i = 0; i < nsm; ++i) a[i] = h[2 * i + (mode == 0 ? 0 : 1)];
      std::sort(a.begin(), a.end());
      med[mode] = (double)a[nsm / 2];
    }
    if (rc != 0) break;
    cudaMemcpy(&st, d_status, 4, cudaMemcpyDeviceToHost);
    out[6] = st ? -1.0 : med[0];
    out[7] = med[1];
    out[8] = st ? -1.0 : med[2];
  } while (false);
  if (d_out) cudaFree(d_out);
  if (d_cyc) cudaFree(d_cyc);
  if (d_cnt) cudaFree(d_cnt);
  if (d_status) cudaFree(d_status);
  return rc;
}
