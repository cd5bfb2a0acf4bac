// walk_kernel.cuh — the walk-resident megakernel for the serial draft head (sm_103a).
//
// "Weights That Stay: On-Chip Megakernels for Serial Heads in Speculative Decoding":
//  - abstract / Fig. 1: each SM keeps a shard of W for the whole walk and only tokens or state cross
//    between steps;
//  - Fig. 2: every step projects the state through the same vocabulary projection W and the chosen
//    token drives the next step;
//  - Fig. 7: the projection is added to the base logits and rounded once;
//  - Fig. 8: each CTA scores its rows, packs its local winner, atomically updates the maximum key and an
//    arrival count, waits for all CTAs and uses the common winner.
//
// Design on GB300 (one persistent cooperative CTA of 384 threads per SM):
//  - W is split into 16-row groups. Each CTA owns `ng` consecutive groups and keeps them in three
//    on-chip tiers for the whole walk: shared memory, tensor memory (written once with tcgen05.st, read
//    every step with tcgen05.ld) and registers. The whole shard arrives by TMA (128-byte swizzle) through
//    a ring of the shared-memory slots: they carry the tensor-memory and register groups first, which
//    their warps move on, and then their own groups.
//  - The projection of a group is 16 (r = 256) mma.sync.m16n8k16 bf16 -> fp32 ops whose A operand is
//    the W group and whose B operand holds the bf16 states of up to 8 walks (two ops for 16 walks).
//    The k index inside each 64-wide box is permuted so that one 16-byte shared-memory load gives a
//    thread a full A fragment without bank conflicts; the B fragments use the same permutation, which
//    makes them 32 contiguous bytes of the state.
//  - The fp32 result plus the base logit is the selection key (plus Gumbel noise when T > 0); keys are
//    packed as ord(key) << 32 | (2^32 - 1 - row) so an unsigned 64-bit maximum picks the largest key
//    and the smallest row on ties.
//  - Cross-CTA exchange per step: each CTA stores its winner, tagged with the step, into its own 64-bit
//    slot (a relaxed store) and adds one to a relaxed arrival counter. Once the counter shows all but 64
//    CTAs, the readers poll every slot, re-reading those whose tag is not yet the step's, and reduce; the
//    words carry their own step, so no fence is needed. Several walks are read by several warps at once.
//    Every wait is bounded by a time limit that ends the walk with a status instead of hanging.
//  - State advance on the GPU: Markov u <- E[x]; recurrent h <- tanh(A h + E[x] + c) where each CTA
//    computes a slice of A h during the step (published as tagged words) and every CTA finishes the
//    update redundantly.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <type_traits>

namespace whead {

constexpr int kThreads = 384;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxB = 16;
constexpr int kMaxGamma = 64;
constexpr int kMaxWarpGroups = 32;
constexpr int kMaxGrid = 256;  // CTAs per walk: the exchange reads up to 8 slots per lane of one warp
constexpr int kGroupRows = 16;
constexpr int kBoxBytes = kGroupRows * 128;  // one 16-row x 64-element bf16 box
constexpr int kTmaChunkGroups = 8;           // groups per large TMA copy (128 rows x 64 elements)
constexpr int kMaxStaged = 64;  // staged groups of the ring entry (their barriers sit in the exchange words)
static_assert(kMaxStaged * 12 <= kWarps * kMaxB * 8, "the ring's barriers and flags fit in the exchange words");

// device status codes (match the public WHEAD_ERR_* values)
constexpr int kStatusTimeout = -4;
constexpr int kStatusInternal = -6;

constexpr uint32_t kFlagLogitsF32 = 1u << 0;
constexpr uint32_t kFlagFixedLatent = 1u << 1;
constexpr uint32_t kFlagSkipArrival = 1u << 8;
constexpr uint32_t kFlagBaseAsync = 1u << 24;  // set by the library: next step's base logits copied during a step

struct WalkArgs {
  const uint16_t* W;  // rows of rw 16-bit words: bf16 values, or (E4M3 weights) pairs of 8-bit codes
  const float* sw;    // E4M3 weights: one fp32 scale per row of W; null otherwise
  const uint16_t* E;
  const float* A;
  const float* c;
  const float* base;
  const float* s0;
  int32_t* tokens;
  unsigned long long* keys;  // optional: each step's winning packed key per walk, ord(key) << 32 | ~row
  void* logits;
  float* state;
  unsigned long long* slots;        // [2 step parities][B][grid] tagged keys for this call (walk-major)
  unsigned int* cnt;                // arrival counter for this call
  unsigned long long* slots_reset;  // the other call parity (or null): cleared during this call
  unsigned int* cnt_reset;
  int32_t slots_reset_count;        // words to clear at slots_reset
  unsigned long long* ah;           // [2 step parities][B][r]: slices of A h exchanged between CTAs, each word
                                    // (t + 1) << 32 | fp32 bits, written relaxed and read until the tag is step t's
  unsigned long long* ah_reset;     // the other call parity's slices (or null): cleared during this call
  int32_t ah_reset_count;           // words to clear at ah_reset
  int* status;
  unsigned long long* trace;  // optional phase stamps: [grid][trace_stride] (clock64 half, globaltimer half)
  int32_t trace_stride;
  int64_t V;
  int64_t v_offset;  // global index of W's first row (a vocabulary shard); a multiple of 16
  int64_t t0;
  uint64_t seed;
  uint64_t timeout_ns;
  float T;
  int32_t r;
  int32_t rw;        // length of a row of W in 16-bit words: r, or r / 2 for E4M3 codes
  int32_t B;
  int32_t gamma;
  int32_t kind;
  uint32_t flags;
  int32_t ng;        // groups per CTA
  int32_t n_smem;    // local groups [0, n_smem) live in shared memory
  int32_t n_tmem;    // [n_smem, n_smem + n_tmem) in tensor memory
  int32_t n_rf;      // then in registers (at most one per warp)
  int32_t n_stream;  // the rest are re-read from global memory (L2) every step
  uint32_t tmem_cols;
  int32_t smem_w_bytes;
  int32_t ra;        // recurrent: rows of A per CTA
  uint32_t rf_warp_mask;  // warps that keep one group in registers (they own no tensor-memory group)
  int32_t ah_warp;        // recurrent: the warp (never a register warp) that computes the CTA's slice of A h
  int32_t wl_count[kWarps];
  // work list of each warp: bits 0..7 CTA-local group, bits 8..9 tier, bits 16..25 tensor-memory column
  uint32_t wl[kWarps][kMaxWarpGroups];
};

constexpr uint32_t kTierSmem = 0, kTierTmem = 1, kTierRf = 2, kTierStream = 3;
__host__ __device__ constexpr uint32_t wl_entry(int j, uint32_t tier, int col) {
  return (uint32_t)j | (tier << 8) | ((uint32_t)col << 16);
}

// Shared-memory layout after the W tier (byte offsets from the 1024-aligned base).
struct SmemLayout {
  int red, win, misc, base, h, a, sw, q, qs, total;
  __host__ __device__ static SmemLayout make(int smem_w_bytes, int B, int r, int ra, bool recurrent, int ng,
                                             bool f8 = false) {
    SmemLayout L;
    L.red = smem_w_bytes;                       // [kWarps][kMaxB] u64
    L.win = L.red + kWarps * kMaxB * 8;         // [kMaxB] int32
    L.misc = L.win + kMaxB * 4;                 // mbarrier u64, tmem addr u32, abort flag u32
    L.base = L.misc + 16;                       // [B][ng * 16] fp32: this step's base logits of the CTA's rows
    L.h = L.base + B * ng * kGroupRows * 4;     // recurrent: [B][r] fp32
    L.a = L.h + (recurrent ? B * r * 4 : 0);    // recurrent: [ra][r] fp32
    L.sw = L.a + (recurrent ? ra * r * 4 : 0);  // E4M3 weights: [ng * 16] fp32 row scales
    L.q = L.sw + (f8 ? ng * kGroupRows * 4 : 0);  // E4M3: [2B][r + 16] codes of each walk's hi and lo vectors
    L.qs = L.q + (f8 ? 2 * B * (r + 16) : 0);     // E4M3: [2B] fp32 scales of those vectors
    L.total = L.qs + (f8 ? 2 * kMaxB * 4 : 0);
    return L;
  }
};

// Shared memory for the incoming base-logit buffer of asynchronous base copies (16 bytes of alignment slack).
__host__ __device__ inline int base_in_bytes(int B, int ng) { return 16 + B * ng * kGroupRows * 4; }

// ------------------------------------------------------------------------------------------------
// small device helpers
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Phase stamp k of this CTA (thread 0 only): SM clock in the first half of the CTA's row, global
// nanosecond timer in the second half.
__device__ __forceinline__ void trace_stamp(const WalkArgs& P, int k) {
  if (P.trace != nullptr && threadIdx.x == 0) {
    unsigned long long* row = P.trace + (int64_t)blockIdx.x * P.trace_stride;
    row[k] = (unsigned long long)clock64();
    row[P.trace_stride / 2 + k] = globaltimer_ns();
  }
}
constexpr int kTraceStampsPerStep = 4;
__host__ __device__ constexpr int trace_stride_for(int max_gamma) { return 2 * (2 + kTraceStampsPerStep * max_gamma); }

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same op with a zero accumulator input (starts a sum without zeroing registers first).
__device__ __forceinline__ void mma_bf16_16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                 uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// f16 x f16 -> fp32, 16 x 8 x 16 (used for E4M3 data, which f16 holds exactly).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16_16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// Four E4M3 codes (one word) to two f16x2 words: .x from bytes 0 and 1, .y from bytes 2 and 3 (exact).
__device__ __forceinline__ uint2 e4m3x4_to_f16(uint32_t w) {
  uint32_t lo, hi;
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.rn.f16x2.e4m3x2 %0, l;\n cvt.rn.f16x2.e4m3x2 %1, h;\n}\n"
      : "=r"(lo), "=r"(hi) : "r"(w));
  return make_uint2(lo, hi);
}

// E4M3 x E4M3 -> fp32, 16 x 8 x 32. Its fragments have the bf16 16 x 8 x 16 layout byte for byte (each 32-bit
// register holds four 8-bit values where the bf16 layout holds two 16-bit ones), so the same storage orders
// serve both formats.
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_e4m3_16832_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                 uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ void tmem_ld16(uint32_t (&a)[16], uint32_t taddr) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
        "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15])
      : "r"(taddr));
}

// 32 columns of this warp's lane quadrant: two boxes of one group.
__device__ __forceinline__ void tmem_ld32(uint32_t (&a)[2][16], uint32_t taddr) {
#define WH_R16(b) "=r"(a[b][0]), "=r"(a[b][1]), "=r"(a[b][2]), "=r"(a[b][3]), "=r"(a[b][4]), "=r"(a[b][5]), \
    "=r"(a[b][6]), "=r"(a[b][7]), "=r"(a[b][8]), "=r"(a[b][9]), "=r"(a[b][10]), "=r"(a[b][11]), "=r"(a[b][12]), \
    "=r"(a[b][13]), "=r"(a[b][14]), "=r"(a[b][15])
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : WH_R16(0), WH_R16(1)
      : "r"(taddr));
#undef WH_R16
}

// 64 columns of this warp's lane quadrant: the four boxes of one group in a single load.
__device__ __forceinline__ void tmem_ld64(uint32_t (&a)[4][16], uint32_t taddr) {
#define WH_R16(b) "=r"(a[b][0]), "=r"(a[b][1]), "=r"(a[b][2]), "=r"(a[b][3]), "=r"(a[b][4]), "=r"(a[b][5]), \
    "=r"(a[b][6]), "=r"(a[b][7]), "=r"(a[b][8]), "=r"(a[b][9]), "=r"(a[b][10]), "=r"(a[b][11]), "=r"(a[b][12]), \
    "=r"(a[b][13]), "=r"(a[b][14]), "=r"(a[b][15])
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : WH_R16(0), WH_R16(1), WH_R16(2), WH_R16(3)
      : "r"(taddr));
#undef WH_R16
}

// Waits for this thread's tcgen05.ld; the registers are tied to the wait so no use is scheduled before it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&a)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
                 "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]),
                 "+r"(a[15])
               :
               : "memory");
}

// Waits for all of this thread's tcgen05.ld and ties every box's registers to the wait.
template <int KB>
__device__ __forceinline__ void tmem_wait_ld_boxes(uint32_t (&a)[KB][16]) {
  tmem_wait_ld(a[0]);
#pragma unroll
  for (int bx = 1; bx < KB; ++bx)
    asm volatile(""
                 : "+r"(a[bx][0]), "+r"(a[bx][1]), "+r"(a[bx][2]), "+r"(a[bx][3]), "+r"(a[bx][4]), "+r"(a[bx][5]),
                   "+r"(a[bx][6]), "+r"(a[bx][7]), "+r"(a[bx][8]), "+r"(a[bx][9]), "+r"(a[bx][10]), "+r"(a[bx][11]),
                   "+r"(a[bx][12]), "+r"(a[bx][13]), "+r"(a[bx][14]), "+r"(a[bx][15]));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&a)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      :
      : "r"(taddr), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]),
        "r"(a[8]), "r"(a[9]), "r"(a[10]), "r"(a[11]), "r"(a[12]), "r"(a[13]), "r"(a[14]), "r"(a[15])
      : "memory");
}

__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11): multipliers 0xD2511F53 / 0xCD9E8D57,
// key increments 0x9E3779B9 / 0xBB67AE85 before every round but the first.
__device__ __forceinline__ uint4 philox4x32_10(uint4 ctr, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    if (i > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * ctr.x, hi0 = __umulhi(0xD2511F53u, ctr.x);
    const uint32_t lo1 = 0xCD9E8D57u * ctr.z, hi1 = __umulhi(0xCD9E8D57u, ctr.z);
    ctr = make_uint4(hi1 ^ ctr.y ^ k0, lo1, hi0 ^ ctr.w ^ k1, lo0);
  }
  return ctr;
}

// Standard Gumbel noise for (seed, walk b, absolute step tau, row v): counter (v/4, tau, b, 0), word v%4,
// U = ((w >> 9) + 0.5) * 2^-23 (exact in fp32), g = -log(-log U).
// Gumbel noise from one Philox output word: U = ((w >> 9) + 1/2) 2^-23 lies strictly inside (0, 1).
__device__ __forceinline__ float gumbel_from_word(uint32_t w) {
  const float u = __fmul_rn(__fadd_rn(__uint2float_rn(w >> 9), 0.5f), 0x1p-23f);
  return -logf(-logf(u));
}

// The four rows 4q .. 4q + 3 of walk b at step tau share one Philox call (counter (q, tau, b, 0)): row v
// takes output word v % 4.
__device__ __forceinline__ uint4 philox_quad(uint64_t seed, uint32_t b, uint32_t tau, uint32_t q) {
  return philox4x32_10(make_uint4(q, tau, b, 0u), (uint32_t)seed, (uint32_t)(seed >> 32));
}

// Order-preserving map of an fp32 key to uint32 (negative: bitwise not; else set the sign bit; -0 -> +0),
// packed above the inverted row so that the unsigned maximum prefers the smaller row on equal keys.
__device__ __forceinline__ unsigned long long pack_key(float key, uint32_t v) {
  uint32_t u = __float_as_uint(key);
  if (u == 0x80000000u) u = 0u;
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (unsigned long long)(0xFFFFFFFFu - v);
}

// Waits on an mbarrier phase with a time limit; returns false if the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t mbar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t_start = globaltimer_ns();
  while (true) {
    uint32_t done;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(done)
                 : "r"(mbar), "r"(parity)
                 : "memory");
    if (done) return true;
    if (globaltimer_ns() - t_start > timeout_ns) return false;
  }
}

// s[i] += x as a shared-memory reduction (no result returned, so the issuing warp does not wait for it).
__device__ __forceinline__ void red_add_shared(float* s, float x) {
  asm volatile("red.shared.add.f32 [%0], %1;" ::"r"(smem_u32(s)), "f"(x) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Warp-wide maximum of a 64-bit value split as (hi, lo): redux.sync on the high words, then on the low words
// of the lanes that hold the maximal high word. Every lane returns the result.
__device__ __forceinline__ unsigned long long warp_max64(uint32_t hi, uint32_t lo) {
  uint32_t mh, ml;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(mh) : "r"(hi));
  const uint32_t l2 = (hi == mh) ? lo : 0u;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(ml) : "r"(l2));
  return ((unsigned long long)mh << 32) | ml;
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) { return a > b ? a : b; }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// Four mma ops of one 64-wide k box (see below). a = [R0 | S0 | R1 | S1]: R rows g, S rows g+8, index 0/1 the two
// 16-byte chunks (2c, 2c+1) of the box. B fragments: 8 registers per box = 16 contiguous bf16 of the state.
// The four ops of a box go to four independent accumulators so that they issue back to back. The box's
// A operands are stored in fragment order: a[4m .. 4m + 3] = {a0, a1, a2, a3} of op m (m = 2 rho + h), so
// each op reads four consecutive registers as they were loaded.
// B fragment words per box: 8 (bf16, or E4M3 codes four to a word), 16 when E4M3 codes are held as f16 pairs.
template <bool F8> constexpr int kBfWords = F8 ? 16 : 8;

template <int KB, int NH, bool F8 = false>
__device__ __forceinline__ void mma_box(float (&acc)[4][NH][4], const uint32_t (&a)[16],
                                        const uint32_t (&bf)[NH][KB][kBfWords<F8>], int bx) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
#pragma unroll
    for (int n = 0; n < NH; ++n) {
      if constexpr (F8) {
        // One 16 x 8 x 32 step on E4M3 codes as two f16 16 x 8 x 16 steps: the first takes the low and the
        // high code pairs of the A words that hold k = 4c .. 4c + 3 (rows g, g + 8) against the same pairs of
        // the B word for those k; the second does the same for k = 16 + 4c .. 16 + 4c + 3. A and B split
        // every 4-value word the same way, so each product meets its partner.
        const uint2 p0 = e4m3x4_to_f16(a[4 * m]), p1 = e4m3x4_to_f16(a[4 * m + 1]);
        const uint2 p2 = e4m3x4_to_f16(a[4 * m + 2]), p3 = e4m3x4_to_f16(a[4 * m + 3]);
        if (bx == 0)
          mma_f16_16816_z(acc[m][n], p0.x, p1.x, p0.y, p1.y, bf[n][bx][4 * m], bf[n][bx][4 * m + 1]);
        else
          mma_f16_16816(acc[m][n], p0.x, p1.x, p0.y, p1.y, bf[n][bx][4 * m], bf[n][bx][4 * m + 1]);
        mma_f16_16816(acc[m][n], p2.x, p3.x, p2.y, p3.y, bf[n][bx][4 * m + 2], bf[n][bx][4 * m + 3]);
      } else {
        if (bx == 0)
          mma_bf16_16816_z(acc[m][n], a[4 * m], a[4 * m + 1], a[4 * m + 2], a[4 * m + 3], bf[n][bx][2 * m],
                           bf[n][bx][2 * m + 1]);
        else
          mma_bf16_16816(acc[m][n], a[4 * m], a[4 * m + 1], a[4 * m + 2], a[4 * m + 3], bf[n][bx][2 * m],
                         bf[n][bx][2 * m + 1]);
      }
    }
  }
}

// ---- E4M3 weights: the state as two scaled E4M3 vectors -----------------------------------------------------
// (Fig. 7 of the pages represents u by two 8-bit vectors whose scaled projections are summed.)

// Four fp32 values to four E4M3 codes (round to nearest even, saturating at +-448), first value in byte 0.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

__device__ __forceinline__ float e4m3_value(uint32_t code) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3)));
}

// Largest |x| over the warp (non-negative floats order as their bit patterns), every lane gets it.
__device__ __forceinline__ float warp_absmax(float m) {
  uint32_t b = __float_as_uint(fabsf(m)), r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(b));
  return __uint_as_float(r);
}

// Quantizes a vector spread over the warp (lane L holds elements [L * EPL, L * EPL + EPL)): scale
// s = max|x| / 448, inv = 1 / s (both correctly rounded), codes E4M3(x * inv) packed four to a word. A vector
// whose largest magnitude is below 448 * FLT_MIN (inv would not be finite) gets s = 0 and zero codes.
template <int EPL>
__device__ __forceinline__ float quantize_e4m3_warp(const float (&x)[EPL], uint32_t (&q)[EPL / 4]) {
  const float amax = [&] {
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) m = fmaxf(m, fabsf(x[e]));
    return warp_absmax(m);
  }();
  const bool zero = !(amax >= 448.f * 1.17549435e-38f);
  const float s = zero ? 0.f : __fdiv_rn(amax, 448.f);
  const float inv = zero ? 0.f : __frcp_rn(s);
#pragma unroll
  for (int w = 0; w < EPL / 4; ++w)
    q[w] = zero ? 0u
                : e4m3x4(__fmul_rn(x[4 * w], inv), __fmul_rn(x[4 * w + 1], inv), __fmul_rn(x[4 * w + 2], inv),
                         __fmul_rn(x[4 * w + 3], inv));
  return s;
}

// Warp routine: splits each walk's state into two E4M3 vectors (hi, and the residual lo) and stores them in
// shared memory: row 2w (hi) and 2w + 1 (lo) of s_q (rows of r + 16 bytes, so that the rows a warp reads at
// once start on different banks), scales s_qs[2w], s_qs[2w + 1]. load(w, x) puts walk w's state elements
// [lane * EPL, lane * EPL + EPL) in x. Every lane of the warp must call this.
template <int KB, typename Load>
__device__ __forceinline__ void split_state_smem(uint8_t* s_q, float* s_qs, int B, int r, int lane, Load load) {
  constexpr int EPL = 4 * KB;  // r = 128 KB elements over 32 lanes
  for (int w = 0; w < B; ++w) {
    float x[EPL];
    load(w, x);
    uint32_t qh[KB], ql[KB];
    const float s1 = quantize_e4m3_warp<EPL>(x, qh);
    float res[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const uint32_t code = (qh[e / 4] >> (8 * (e % 4))) & 0xFFu;
      res[e] = __fsub_rn(x[e], __fmul_rn(s1, e4m3_value(code)));
    }
    const float s2 = quantize_e4m3_warp<EPL>(res, ql);
    uint32_t* dh = reinterpret_cast<uint32_t*>(s_q + (2 * w) * (r + 16) + lane * EPL);
    uint32_t* dl = reinterpret_cast<uint32_t*>(s_q + (2 * w + 1) * (r + 16) + lane * EPL);
#pragma unroll
    for (int k = 0; k < KB; ++k) {
      dh[k] = qh[k];
      dl[k] = ql[k];
    }
    if (lane == 0) {
      s_qs[2 * w] = s1;
      s_qs[2 * w + 1] = s2;
    }
  }
}

// B fragments of the E4M3 projection for B <= 4 walks, from the split state in shared memory: column 2w holds
// walk w's hi vector, column 2w + 1 its lo vector, so lane (g, c) reads row g; fragment word i of box bx is
// bytes 128 bx + 32 c + 4 i of that row (the bf16 path's order). s1c / s2c: the scales of walk c, whose sums
// this lane's accumulator columns 2c and 2c + 1 hold.
template <int KB>
__device__ __forceinline__ void bfrag_from_split_smem(uint32_t (&bf)[1][KB][16], float& s1c, float& s2c,
                                                      const uint8_t* s_q, const float* s_qs, int B, int r, int lane) {
  const int g = lane >> 2, c = lane & 3;
  const bool live = (g >> 1) < B;
  const uint8_t* row = s_q + g * (r + 16);
#pragma unroll
  for (int bx = 0; bx < KB; ++bx) {
    uint4 x0 = make_uint4(0u, 0u, 0u, 0u), x1 = x0;
    if (live) {
      const uint4* p = reinterpret_cast<const uint4*>(row + 128 * bx + 32 * c);
      x0 = p[0];
      x1 = p[1];
    }
    // code word i becomes f16 words 2i (its codes 0, 1) and 2i + 1 (codes 2, 3)
    const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint2 h = e4m3x4_to_f16(w[i]);
      bf[0][bx][2 * i] = h.x;
      bf[0][bx][2 * i + 1] = h.y;
    }
  }
  s1c = c < B ? s_qs[2 * c] : 0.f;
  s2c = c < B ? s_qs[2 * c + 1] : 0.f;
}


// Rows g / g + 8 of a box as loaded ([R0 | S0 | R1 | S1]: chunk 2c then 2c + 1 of each row) to fragment
// order: op m = 2 rho + h takes {R_rho[2h], S_rho[2h], R_rho[2h + 1], S_rho[2h + 1]}.
__device__ __forceinline__ void rows_to_fragments(uint32_t (&q)[16], const uint32_t (&a)[16]) {
#pragma unroll
  for (int rho = 0; rho < 2; ++rho)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int m = 2 * rho + h;
      q[4 * m + 0] = a[8 * rho + 2 * h];
      q[4 * m + 1] = a[8 * rho + 4 + 2 * h];
      q[4 * m + 2] = a[8 * rho + 2 * h + 1];
      q[4 * m + 3] = a[8 * rho + 4 + 2 * h + 1];
    }
}

// A fragments of box bx of a group read straight from W in global memory (row-major, unswizzled):
// row g then row g+8, 32 contiguous bytes each (chunks 2c and 2c+1 of the box). Rows >= V read as zero.
__device__ __forceinline__ void load_box_global(uint32_t (&a)[16], const uint16_t* W, int64_t v0, int64_t V, int r,
                                                int bx, int c) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int64_t v = v0 + 8 * half;
    uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
    if (v < V) {
      const uint4* p = reinterpret_cast<const uint4*>(W + v * r + 64 * bx + 16 * c);
      x0 = __ldg(p);
      x1 = __ldg(p + 1);
    }
    // layout [R0 | S0 | R1 | S1]
    a[4 * half + 0] = x0.x; a[4 * half + 1] = x0.y; a[4 * half + 2] = x0.z; a[4 * half + 3] = x0.w;
    a[8 + 4 * half + 0] = x1.x; a[8 + 4 * half + 1] = x1.y; a[8 + 4 * half + 2] = x1.z; a[8 + 4 * half + 3] = x1.w;
  }
}

// Box bx of a group read from global memory straight into fragment order (rows >= V read as zero).
__device__ __forceinline__ void load_box_global_frag(uint32_t (&q)[16], const uint16_t* W, int64_t v0, int64_t V, int r,
                                                     int bx, int c) {
  uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0, y0 = x0, y1 = x0;
  if (v0 < V) {
    const uint4* p = reinterpret_cast<const uint4*>(W + v0 * r + 64 * bx + 16 * c);
    x0 = __ldg(p);
    x1 = __ldg(p + 1);
  }
  if (v0 + 8 < V) {
    const uint4* p = reinterpret_cast<const uint4*>(W + (v0 + 8) * r + 64 * bx + 16 * c);
    y0 = __ldg(p);
    y1 = __ldg(p + 1);
  }
  // x: row g chunks 2c (x0) and 2c + 1 (x1); y: row g + 8. Op m = 2 rho + h takes {R[2h], S[2h], R[2h+1], S[2h+1]}.
  q[0] = x0.x; q[1] = y0.x; q[2] = x0.y; q[3] = y0.y;
  q[4] = x0.z; q[5] = y0.z; q[6] = x0.w; q[7] = y0.w;
  q[8] = x1.x; q[9] = y1.x; q[10] = x1.y; q[11] = y1.y;
  q[12] = x1.z; q[13] = y1.z; q[14] = x1.w; q[15] = y1.w;
}

// Builds the B fragments of walk n from an fp32 state row (global or shared), rounding to bf16.
template <int KB>
__device__ __forceinline__ void bfrag_from_f32(uint32_t (&bf)[KB][8], const float* s, int c) {
#pragma unroll
  for (int bx = 0; bx < KB; ++bx) {
    const float4* p = reinterpret_cast<const float4*>(s + 64 * bx + 16 * c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 f = p[i];
      bf[bx][2 * i] = pack_bf16x2(f.x, f.y);
      bf[bx][2 * i + 1] = pack_bf16x2(f.z, f.w);
    }
  }
}

template <int KB>
__device__ __forceinline__ void bfrag_from_bf16_row(uint32_t (&bf)[KB][8], const uint16_t* e, int c) {
#pragma unroll
  for (int bx = 0; bx < KB; ++bx) {
    const uint4* p = reinterpret_cast<const uint4*>(e + 64 * bx + 16 * c);
    const uint4 x0 = __ldg(p), x1 = __ldg(p + 1);
    bf[bx][0] = x0.x; bf[bx][1] = x0.y; bf[bx][2] = x0.z; bf[bx][3] = x0.w;
    bf[bx][4] = x1.x; bf[bx][5] = x1.y; bf[bx][6] = x1.z; bf[bx][7] = x1.w;
  }
}

// Copies the base logits of step t for this CTA's rows into shared memory (coalesced; rows >= V read as
// zero) using threads [first, first + count), and asks L2 for the rows of step t + 1. The base logits may
// sit in host memory that the GPU reads in place; the L2 request one step ahead hides that latency too.
__device__ __forceinline__ void stage_base(const WalkArgs& P, float* s_base, int64_t row_base, int t, int first,
                                           int count) {
  const int rows = P.ng * kGroupRows;
  const int i0 = (int)threadIdx.x - first;
  if (i0 < 0 || i0 >= count || t >= P.gamma) return;
  const int valid = (int)min((int64_t)rows, P.V - row_base);  // rows of this CTA below V (may be <= 0)
  // (walk, row) pairs flattened; each thread issues four loads before it stores any of them, so their
  // latencies overlap instead of adding up
  const int total = P.B * rows;
  for (int i = i0; i < total; i += 4 * count) {
    float x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = i + u * count, n = k / rows, lr = k - n * rows;
      x[u] = (k < total && lr < valid) ? __ldg(P.base + ((int64_t)n * P.gamma + t) * P.V + row_base + lr) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * count < total) s_base[i + u * count] = x[u];
  }
  if (t + 1 < P.gamma)
    for (int n = 0; n < P.B; ++n) {
      const float* nxt = P.base + ((int64_t)n * P.gamma + t + 1) * P.V + row_base;
      for (int lr = 32 * i0; lr < valid; lr += 32 * count) prefetch_l2(nxt + lr);
    }
}

// The same rows as stage_base, copied with cp.async so that no thread waits for them here: 16 bytes per copy
// when every row of base starts on a 16-byte boundary (rows past V zero-filled by the copy's source size), else
// 4 bytes per copy. The caller runs cp.async.wait_all before the rows are read. Also asks L2 for step t + 1.
__device__ __forceinline__ void stage_base_cp(const WalkArgs& P, float* s_base, int64_t row_base, int t, int first,
                                              int count) {
  const int rows = P.ng * kGroupRows;
  const int i0 = (int)threadIdx.x - first;
  if (i0 < 0 || i0 >= count || t >= P.gamma) return;
  const int valid = (int)min((int64_t)rows, P.V - row_base);  // rows of this CTA below V (may be <= 0)
  if ((P.V & 3) == 0 && (reinterpret_cast<uintptr_t>(P.base) & 15u) == 0) {
    const int chunks = rows / 4;  // rows is a multiple of 16
    for (int i = i0; i < P.B * chunks; i += count) {
      const int n = i / chunks, lr = 4 * (i - n * chunks);
      const int nbytes = 4 * max(0, min(4, valid - lr));
      // a copy with no source bytes still names an address inside base
      const float* src = nbytes ? P.base + ((int64_t)n * P.gamma + t) * P.V + row_base + lr : P.base;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(s_base + n * rows + lr)), "l"(src),
                   "r"(nbytes)
                   : "memory");
    }
  } else {
    for (int i = i0; i < P.B * rows; i += count) {
      const int n = i / rows, lr = i - n * rows;
      if (lr < valid)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(s_base + i)),
                     "l"(P.base + ((int64_t)n * P.gamma + t) * P.V + row_base + lr)
                     : "memory");
      else
        s_base[i] = 0.f;
    }
  }
  if (t + 1 < P.gamma)
    for (int n = 0; n < P.B; ++n) {
      const float* nxt = P.base + ((int64_t)n * P.gamma + t + 1) * P.V + row_base;
      for (int lr = 32 * i0; lr < valid; lr += 32 * count) prefetch_l2(nxt + lr);
    }
}

// The same rows as stage_base, copied asynchronously into a second buffer (cp.async, 4 bytes per row; the
// group is committed here and waited for by the same thread with cp.async.wait_all). Used when the base
// logits sit behind a slow link (host memory read in place): the copy for step t + 2 is issued during step t,
// so a whole step passes before its rows are needed.
__device__ __forceinline__ void copy_base_async(const WalkArgs& P, float* s_dst, int64_t row_base, int t, int first,
                                                int count) {
  const int rows = P.ng * kGroupRows;
  const int i0 = (int)threadIdx.x - first;
  if (i0 < 0 || i0 >= count || t >= P.gamma) return;
  const int valid = (int)min((int64_t)rows, P.V - row_base);
  for (int n = 0; n < P.B; ++n) {
    const float* src = P.base + ((int64_t)n * P.gamma + t) * P.V + row_base;
    float* dst = s_dst + n * rows;
    for (int lr = i0; lr < rows; lr += count) {
      if (lr < valid)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst + lr)), "l"(src + lr) : "memory");
      else
        dst[lr] = 0.f;
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Each thread moves the rows it copied with copy_base_async (same partition) into this step's buffer.
__device__ __forceinline__ void move_base(const WalkArgs& P, float* s_base, const float* s_in, int t, int first,
                                          int count) {
  const int rows = P.ng * kGroupRows;
  const int i0 = (int)threadIdx.x - first;
  if (i0 < 0 || i0 >= count || t >= P.gamma) return;
  for (int n = 0; n < P.B; ++n)
    for (int lr = i0; lr < rows; lr += count) s_base[n * rows + lr] = s_in[n * rows + lr];
}

// Several walks: one warp reads every CTA's slot of walk n until each word carries step t's tag (re-reading the
// stale ones; bounded by timeout_ns from t_start) and returns the largest packed key in every lane, or 0 on
// time-out. The warp takes its decision on leaving the loop as a whole.
template <int kSlotsPerLane>
__device__ __forceinline__ unsigned long long read_walk_slots(const unsigned long long* sl, int G, int B, int n, int t,
                                                              int lane, uint64_t t_start, uint64_t timeout_ns,
                                                              bool& late) {
  const unsigned long long tag = (unsigned long long)(t + 1) << 56;
  unsigned long long w[kSlotsPerLane];
#pragma unroll
  for (int i = 0; i < kSlotsPerLane; ++i) w[i] = (lane + 32 * i < G) ? 0ull : tag;  // tag 0: not read yet
  for (uint32_t spins = 0;; ) {
#pragma unroll
    for (int i = 0; i < kSlotsPerLane; ++i) {
      const int cc = lane + 32 * i;
      if (cc < G && (w[i] >> 56) != (unsigned long long)(t + 1))
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w[i]) : "l"(sl + (int64_t)n * G + cc) : "memory");
    }
    bool fresh = true;
#pragma unroll
    for (int i = 0; i < kSlotsPerLane; ++i) fresh = fresh && ((w[i] >> 56) == (unsigned long long)(t + 1));
    if (__all_sync(0xffffffffu, fresh)) break;
    if ((++spins & 15u) == 0u && __any_sync(0xffffffffu, globaltimer_ns() - t_start > timeout_ns)) {
      late = true;
      return 0ull;
    }
  }
  unsigned long long best = 0ull;
#pragma unroll
  for (int i = 0; i < kSlotsPerLane; ++i) best = umax64(best, w[i] & 0x00FFFFFFFFFFFFFFull);
  return warp_max64((uint32_t)(best >> 32), (uint32_t)best);
}

// ------------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------------
// KB: 64-wide boxes of the rank (r = 64 KB). NH: n8 halves of the batch (B <= 8 * NH). NB1: B == 1.
// Warp roles: warps in rf_warp_mask keep one group in registers (plus shared-memory groups); the others
// own the tensor-memory groups of their lane quadrant (plus shared-memory groups). The two roles run
// separately compiled copies of the step loop so that neither pays for the other's registers.
// F8: E4M3 weights. ASYNC: each step's base logits are copied asynchronously a step ahead into a second
// buffer (walks that read them from host memory); kept out of the other variants' step loop. REC: the recurrent
// head (the Markov head's copy carries none of its code: no A h slices, no tanh advance).
template <int KB, int NH, bool NB1, bool F8, bool ASYNC, bool REC>
__global__ void __launch_bounds__(kThreads, 1)
    walk_kernel(const __grid_constant__ CUtensorMap tmapW, const __grid_constant__ CUtensorMap tmapW128,
                const __grid_constant__ WalkArgs P) {
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int G = gridDim.x, cta = blockIdx.x;
  const int r = P.r, B = P.B, gamma = P.gamma;
  const int64_t V = P.V;
  constexpr bool recurrent = REC;  // the host launches the instantiation of the head's kind

  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const SmemLayout L = SmemLayout::make(P.smem_w_bytes, B, r, P.ra, recurrent, P.ng, F8);
  uint8_t* sW = smem;
  unsigned long long* s_red = reinterpret_cast<unsigned long long*>(smem + L.red);
  int32_t* s_win = reinterpret_cast<int32_t*>(smem + L.win);
  unsigned long long* s_mbar = reinterpret_cast<unsigned long long*>(smem + L.misc);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L.misc + 8);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.misc + 12);
  float* s_base = reinterpret_cast<float*>(smem + L.base);
  // with asynchronous base copies, a second buffer past the end of the layout receives the step after next
  constexpr bool base_async = ASYNC;  // launched with kFlagBaseAsync set
  float* s_base_in = reinterpret_cast<float*>(smem + ((L.total + 15) & ~15));
  float* s_h = reinterpret_cast<float*>(smem + L.h);
  float* s_A = reinterpret_cast<float*>(smem + L.a);
  float* s_sw = reinterpret_cast<float*>(smem + L.sw);  // E4M3 weights: scales of this CTA's rows
  uint8_t* s_q = smem + L.q;                            // E4M3 weights: each walk's state as two E4M3 vectors
  float* s_qs = reinterpret_cast<float*>(smem + L.qs);  // and their scales
  static_assert(!F8 || NH == 1, "E4M3 weights take two accumulator columns per walk: at most 4 walks");
  // several walks: the warps read the walks' exchange slots in parallel
  constexpr bool kParRead = !NB1;

  const uint32_t mbar = smem_u32(s_mbar);
  trace_stamp(P, 0);
  const int64_t row_base = (int64_t)cta * P.ng * kGroupRows;
  const int64_t vg_base = P.v_offset + row_base;  // global row of the CTA's first row (keys, noise, tokens)
  const int rows_cta = P.ng * kGroupRows;
  const int my_count = P.wl_count[warp];
  const uint32_t my_entry = (lane < my_count) ? P.wl[warp][lane] : 0u;
  const bool rf_warp = (P.rf_warp_mask >> warp) & 1u;

  // Shard load through a ring: the shared tier's n_smem slots first receive the tensor-memory and register
  // groups, which their owner warps move on, and then their own groups, so that the whole shard streams in by TMA
  // with every slot's copy in flight. Staged group k (local group n_smem + k) passes through slot k % n_smem and
  // completes on barrier k, used for one phase only. The barriers and the issue flags sit in the exchange words,
  // which the walk uses only after the entry. Without a shared tier, or with more than kMaxStaged groups to
  // stage, the tensor-memory and register groups are loaded through registers instead.
  const int n_st = P.n_tmem + P.n_rf;  // staged groups
  const bool ring = P.n_smem > 0 && n_st > 0 && n_st <= kMaxStaged;
  volatile int* s_issued = reinterpret_cast<volatile int*>(s_red + kMaxStaged);  // [n_st] staged copy issued
  auto stage_bar = [&](int k) { return smem_u32(s_red + k); };

  // ---------------- set-up ----------------
  if (tid == 0) {
    *s_abort = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar) : "memory");
    if (ring)
      for (int k = 0; k < n_st; ++k) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(stage_bar(k)) : "memory");
        s_issued[k] = 0;
      }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && P.tmem_cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                 "r"(P.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // clear the exchange words of the other call parity (the previous call on this stream has finished)
  if (cta == G - 1 && P.slots_reset != nullptr) {
    for (int i = tid; i < P.slots_reset_count; i += kThreads) P.slots_reset[i] = 0ull;
    if (tid == 0) *P.cnt_reset = 0u;
  }
  if (cta == G - 1 && P.ah_reset != nullptr)
    for (int i = tid; i < P.ah_reset_count; i += kThreads) P.ah_reset[i] = 0ull;
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem_base = P.tmem_cols ? *s_tmem : 0u;
  const uint32_t lane_quadrant = (uint32_t)(32 * (warp & 3)) << 16;

  // ---------------- entry: load the shard once (Fig. 4: the one-time shard load) ----------------
  // one group (16 rows, KB boxes) into slot s of the shared tier, completing on barrier bar
  auto issue_group = [&](int s, int j, uint32_t bar) {
    const int y = (int)(row_base + (int64_t)kGroupRows * j);
#pragma unroll
    for (int bx = 0; bx < KB; ++bx)
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
              smem_u32(sW) + (uint32_t)(bx * P.n_smem + s) * kBoxBytes),
          "l"(reinterpret_cast<uint64_t>(&tmapW)), "r"(64 * bx), "r"(y), "r"(bar)
          : "memory");
  };
  // the next copy into slot s once staged group k has left it: staged group k + n_smem, else the slot's own group
  auto refill = [&](int s, int k) {
    const int k2 = k + P.n_smem;
    if (k2 < n_st) {
      s_issued[k2] = 1;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(stage_bar(k2)), "r"(KB * kBoxBytes)
                   : "memory");
      issue_group(s, P.n_smem + k2, stage_bar(k2));
    } else {
      issue_group(s, s, mbar);
    }
  };
  if (tid == 0 && ring) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(P.n_smem * KB * kBoxBytes)
                 : "memory");
    for (int s = 0; s < P.n_smem; ++s) refill(s, s - P.n_smem);
  }
  if (tid == 0 && P.n_smem > 0 && !ring) {
    // box-major shared tier: box bx of local group j at (bx * n_smem + j) * 2048. Runs of 8 groups go in one
    // 128-row copy, the remainder in 16-row copies.
    const uint32_t bytes = (uint32_t)(P.n_smem * KB * kBoxBytes);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
    const uint32_t dst0 = smem_u32(sW);
    const int full = P.n_smem / kTmaChunkGroups;
    for (int bx = 0; bx < KB; ++bx) {
      const int x = 64 * bx;
      for (int j = 0; j < P.n_smem;) {
        const uint32_t dst = dst0 + (uint32_t)(bx * P.n_smem + j) * kBoxBytes;
        const int y = (int)(row_base + (int64_t)kGroupRows * j);
        if (j < full * kTmaChunkGroups) {
          asm volatile(
              "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
              "l"(reinterpret_cast<uint64_t>(&tmapW128)), "r"(x), "r"(y), "r"(mbar)
              : "memory");
          j += kTmaChunkGroups;
        } else {
          asm volatile(
              "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
              "l"(reinterpret_cast<uint64_t>(&tmapW)), "r"(x), "r"(y), "r"(mbar)
              : "memory");
          j += 1;
        }
      }
    }
  }
  if (!ring) {
    stage_base(P, s_base, row_base, 0, 0, kThreads);
    if constexpr (base_async) copy_base_async(P, s_base_in, row_base, 1, 32, kThreads - 32);
  }

  // without the ring: the tensor-memory groups of this warp go global -> registers (all boxes of a group in
  // flight) -> tcgen05.st
  if (!rf_warp && !ring) {
    for (int e = 0; e < my_count; ++e) {
      const uint32_t ent = __shfl_sync(0xffffffffu, my_entry, e);
      if (((ent >> 8) & 3u) != kTierTmem) continue;
      const int j = (int)(ent & 0xFFu);
      const uint32_t taddr = tmem_base + lane_quadrant + (ent >> 16);
      const int64_t v0 = row_base + (int64_t)kGroupRows * j + g;
      uint32_t a[KB][16];
#pragma unroll
      for (int bx = 0; bx < KB; ++bx) load_box_global(a[bx], P.W, v0, V, P.rw, bx, c);
#pragma unroll
      for (int bx = 0; bx < KB; ++bx) {
        uint32_t q[16];
        rows_to_fragments(q, a[bx]);
        tmem_st16(taddr + 16 * bx, q);
      }
    }
  }
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  // register-resident group of a register warp (register warps own no tensor-memory group): without the ring its
  // loads are issued here, so they land while the rest of the entry runs; with it, the group comes through a slot
  uint32_t rfA[KB][16];
  if (NH == 1 && rf_warp) {  // the planner gives register groups only to batches of up to 8 walks
    int jr = -1;
    if (!ring)
      for (int e = 0; e < my_count; ++e) {
        const uint32_t ent = __shfl_sync(0xffffffffu, my_entry, e);
        if (((ent >> 8) & 3u) == kTierRf) jr = (int)(ent & 0xFFu);
      }
#pragma unroll
    for (int bx = 0; bx < KB; ++bx) {
      if (jr >= 0) {
        uint32_t a[16];
        load_box_global(a, P.W, row_base + (int64_t)kGroupRows * jr + g, V, P.rw, bx, c);
        rows_to_fragments(rfA[bx], a);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) rfA[bx][i] = 0u;
      }
    }
  }
  // ring: each warp takes its staged groups out of their slots in the order they were issued (staged group k
  // sits in slot k % n_smem in round k / n_smem), then hands the slot on
  if (ring) {
    const uint32_t off0 = (uint32_t)(((2 * c) ^ g) << 4), off1 = (uint32_t)(((2 * c + 1) ^ g) << 4);
    for (int e = 0; e < my_count; ++e) {
      const uint32_t ent = __shfl_sync(0xffffffffu, my_entry, e);
      const uint32_t tier = (ent >> 8) & 3u;
      if (tier != kTierTmem && tier != kTierRf) continue;
      const int k = (int)(ent & 0xFFu) - P.n_smem, sl = k % P.n_smem;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(stage_bar(k), 0u, P.timeout_ns))) {
        if (lane == 0) atomicCAS(P.status, 0, kStatusTimeout);
        *s_abort = 1;
        break;
      }
      const uint32_t taddr = tmem_base + lane_quadrant + (ent >> 16);
#pragma unroll
      for (int bx = 0; bx < KB; ++bx) {
        // the 128-byte-swizzled box: row g's chunks 2c and 2c + 1 and the same chunks of row g + 8
        const uint8_t* box = sW + (uint32_t)(bx * P.n_smem + sl) * kBoxBytes;
        const uint4 r0 = *reinterpret_cast<const uint4*>(box + g * 128 + off0);
        const uint4 s0 = *reinterpret_cast<const uint4*>(box + (g + 8) * 128 + off0);
        const uint4 r1 = *reinterpret_cast<const uint4*>(box + g * 128 + off1);
        const uint4 s1 = *reinterpret_cast<const uint4*>(box + (g + 8) * 128 + off1);
        const uint32_t a[16] = {r0.x, r0.y, r0.z, r0.w, s0.x, s0.y, s0.z, s0.w,
                                r1.x, r1.y, r1.z, r1.w, s1.x, s1.y, s1.z, s1.w};
        if (tier == kTierTmem) {
          uint32_t q[16];
          rows_to_fragments(q, a);
          tmem_st16(taddr + 16 * bx, q);
        } else if (NH == 1) {
          rows_to_fragments(rfA[bx], a);
        }
      }
      __syncwarp();
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        refill(sl, k);
      }
      __syncwarp();
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    stage_base(P, s_base, row_base, 0, 0, kThreads);
    if constexpr (base_async) copy_base_async(P, s_base_in, row_base, 1, 32, kThreads - 32);
  }
  // streamed groups: ask L2 for their rows now, so that every step reads them from L2
  for (int e = 0; e < my_count; ++e) {
    const uint32_t ent = __shfl_sync(0xffffffffu, my_entry, e);
    if (((ent >> 8) & 3u) != kTierStream) continue;
    // the group's 16 rows are 32 rw contiguous bytes: one prefetch per 128-byte line, rows below V only
    const int64_t v0 = row_base + (int64_t)kGroupRows * (int)(ent & 0xFFu);
    const uint8_t* gb = reinterpret_cast<const uint8_t*>(P.W + v0 * P.rw);
    for (int L = lane; L < P.rw / 4; L += 32)
      if (v0 + (L * 128) / (2 * P.rw) < V) prefetch_l2(gb + L * 128);
  }

  // E4M3 weights: the row scales of this CTA's rows (rows past V read as zero)
  if constexpr (F8)
    for (int lr = tid; lr < rows_cta; lr += kThreads) s_sw[lr] = (row_base + lr < V) ? P.sw[row_base + lr] : 0.f;

  // recurrent head: the initial state and this CTA's rows of A
  const int a_lo = cta * P.ra;
  if (recurrent) {
    for (int i = tid; i < B * r; i += kThreads) s_h[i] = P.s0[i];
    for (int i = tid; i < P.ra * r; i += kThreads) {
      const int row = a_lo + i / r;
      s_A[i] = (row < r) ? P.A[(int64_t)row * r + (i % r)] : 0.f;
    }
  }

  // wait for the TMA copies (bounded)
  bool tma_done = true;
  if (P.n_smem > 0) {
    tma_done = __all_sync(0xffffffffu, mbar_wait_bounded(mbar, 0u, P.timeout_ns));
    if (!tma_done) {
      if (tid == 0) atomicCAS(P.status, 0, kStatusTimeout);
      *s_abort = 1;
    }
  }
  // each warp turns whole boxes of the shared tier from the TMA layout (16 rows x 128 B, 128-byte swizzle:
  // chunk ^ (row % 8)) into fragment order; a box is read completely into registers before it is rewritten
  if (tma_done) {
    const uint32_t off0 = (uint32_t)(((2 * c) ^ g) << 4), off1 = (uint32_t)(((2 * c + 1) ^ g) << 4);
    for (int b = warp; b < P.n_smem * KB; b += kWarps) {
      uint8_t* box = sW + (uint32_t)b * kBoxBytes;
      const uint4 r0 = *reinterpret_cast<const uint4*>(box + g * 128 + off0);
      const uint4 s0 = *reinterpret_cast<const uint4*>(box + (g + 8) * 128 + off0);
      const uint4 r1 = *reinterpret_cast<const uint4*>(box + g * 128 + off1);
      const uint4 s1 = *reinterpret_cast<const uint4*>(box + (g + 8) * 128 + off1);
      __syncwarp();
      uint4* out = reinterpret_cast<uint4*>(box) + lane;
      out[0] = make_uint4(r0.x, s0.x, r0.y, s0.y);
      out[32] = make_uint4(r0.z, s0.z, r0.w, s0.w);
      out[64] = make_uint4(r1.x, s1.x, r1.y, s1.y);
      out[96] = make_uint4(r1.z, s1.z, r1.w, s1.w);
    }
  }
  // E4M3 weights: warp 0 splits the initial states into two E4M3 vectors each (read by every warp after
  // the barrier)
  if constexpr (F8) {
    if (warp == 0)
      split_state_smem<KB>(s_q, s_qs, B, r, lane, [&](int w, auto& x) {
        const float* src = P.s0 + (int64_t)w * r + lane * 4 * KB;
#pragma unroll
        for (int e = 0; e < 4 * KB; ++e) x[e] = src[e];
      });
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  // the slot barriers' words become exchange words again (first written after the first step's projection and
  // barrier)
  if (ring) {
    if (!*s_abort) {
      if (tid < n_st) asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(stage_bar(tid)) : "memory");
    } else if (tid == 0) {
      // a wait of the entry timed out: copies still in flight land before the walk is skipped and the CTA exits
      for (int k = 0; k < n_st; ++k)
        if (s_issued[k]) (void)mbar_wait_bounded(stage_bar(k), 0u, P.timeout_ns);
    }
  }
  trace_stamp(P, 1);

  const uint8_t* sW_c = sW;
  const uint32_t box_stride = (uint32_t)(P.n_smem * kBoxBytes);
  const float T = P.T;
  const bool sampled = T > 0.0f;
  const bool t_is_one = T == 1.0f;  // z / 1 is z exactly: the correctly rounded division is skipped
  const bool want_f32 = (P.flags & kFlagLogitsF32) != 0u;

  // ---------------- the walk ----------------
  auto walk = [&](auto rf_tag) {
    constexpr bool RFW = decltype(rf_tag)::value;

    uint32_t bf[NH][KB][kBfWords<F8>];
    // E4M3 weights: the scales of walk c's two state vectors (this lane's accumulator columns 2c, 2c + 1)
    float es1 = 0.f, es2 = 0.f;
    if constexpr (F8) {
      bfrag_from_split_smem<KB>(bf, es1, es2, s_q, s_qs, B, r, lane);
    } else {
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const int n = 8 * h + g;
        if (n < B) {
          bfrag_from_f32<KB>(bf[h], recurrent ? (s_h + n * r) : (P.s0 + (int64_t)n * r), c);
        } else {
#pragma unroll
          for (int bx = 0; bx < KB; ++bx)
#pragma unroll
            for (int i = 0; i < 8; ++i) bf[h][bx][i] = 0u;
        }
      }
    }

    // E4M3 weights, Markov: warp 0 splits each winner's E row into two E4M3 vectors in shared memory
    auto split_winner_rows = [&]() {
      split_state_smem<KB>(s_q, s_qs, B, r, lane, [&](int w, auto& x) {
        const int32_t xw = s_win[w];
        uint32_t u[2 * KB];
#pragma unroll
        for (int e = 0; e < 2 * KB; ++e) u[e] = 0u;
        if ((int64_t)xw >= P.v_offset && (int64_t)xw < P.v_offset + V) {
          const uint16_t* er = P.E + (int64_t)xw * r + lane * 4 * KB;
          if constexpr (KB == 2) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(er));
            u[0] = v.x; u[1] = v.y; u[2] = v.z; u[3] = v.w;
          } else {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(er));
            u[0] = v.x; u[1] = v.y;
          }
        }
#pragma unroll
        for (int e = 0; e < 2 * KB; ++e) {
          x[2 * e] = __uint_as_float(u[e] << 16);
          x[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
        }
      });
    };

    for (int t = 0; t < gamma; ++t) {
      if (*s_abort) break;
      const uint32_t tau = (uint32_t)(P.t0 + t);
      trace_stamp(P, 2 + kTraceStampsPerStep * t);

      // recurrent: this CTA's slice of A h_t, published during the step by the least-loaded warp that keeps no
      // register group (so the register warps' copy of the loop does not carry this code)
      if (!RFW && recurrent && warp == P.ah_warp) {
        for (int p = 0; p < B * P.ra; ++p) {
          const int n = p / P.ra, i = p % P.ra;
          if (a_lo + i >= r) continue;
          // r = kRank is known at compile time: the loads of a row all issue before its chain of fma
          constexpr int kRank = (F8 ? 128 : 64) * KB;
          float s = 0.f;
#pragma unroll
          for (int k = lane; k < kRank; k += 32) s = fmaf(s_A[i * kRank + k], s_h[n * kRank + k], s);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
          if (lane == 0) {
            const unsigned long long word = ((unsigned long long)(t + 1) << 32) | __float_as_uint(s);
            asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(P.ah + ((int64_t)(t & 1) * B + n) * r + a_lo + i),
                         "l"(word)
                         : "memory");
          }
        }
      }

      // the next group's work-list entry and this group's base logits are read a group ahead / at the start, so
      // neither latency sits between a group's last mma and its epilogue
      uint32_t ent_next = __shfl_sync(0xffffffffu, my_entry, 0);
      for (int e = 0; e < my_count; ++e) {
        const uint32_t ent = ent_next;
        ent_next = __shfl_sync(0xffffffffu, my_entry, (e + 1) & 31);
        const int j = (int)(ent & 0xFFu);
        const uint32_t tier = (ent >> 8) & 3u;
        float zb0 = 0.f, zb1 = 0.f;
        if constexpr (NB1) {
          zb0 = s_base[kGroupRows * j + g];
          zb1 = s_base[kGroupRows * j + g + 8];
        }

        float acc[4][NH][4];
        if (tier == kTierSmem) {
          // box-major shared tier (box bx of group j at (bx * n_smem + j) * 2048), each box stored as four
          // lane-major 512-byte fragment blocks: one conflict-free 16-byte load per op
          const uint8_t* p = sW_c + (uint32_t)j * kBoxBytes + (uint32_t)lane * 16u;
#pragma unroll
          for (int bx = 0; bx < KB; ++bx) {
            uint32_t a[16];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const uint4 x = *reinterpret_cast<const uint4*>(p + bx * box_stride + m * 512);
              a[4 * m] = x.x; a[4 * m + 1] = x.y; a[4 * m + 2] = x.z; a[4 * m + 3] = x.w;
            }
            mma_box<KB, NH, F8>(acc, a, bf, bx);
          }
        } else if (tier == kTierTmem) {
          if constexpr (!RFW) {
            const uint32_t taddr = tmem_base + lane_quadrant + (ent >> 16);
            if constexpr (KB == 4 && NH == 1) {
              uint32_t a0[2][16], a1[2][16];
              tmem_ld32(a0, taddr);
              tmem_wait_ld_boxes<2>(a0);
              tmem_ld32(a1, taddr + 32);
              mma_box<KB, NH, F8>(acc, a0[0], bf, 0);
              mma_box<KB, NH, F8>(acc, a0[1], bf, 1);
              tmem_wait_ld_boxes<2>(a1);
              mma_box<KB, NH, F8>(acc, a1[0], bf, 2);
              mma_box<KB, NH, F8>(acc, a1[1], bf, 3);
            } else {
              // boxes read per wait: all of them for one batch half, two when both halves are live
              constexpr int TB = (NH == 1 || KB < 4) ? KB : 2;
#pragma unroll
              for (int b0 = 0; b0 < KB; b0 += TB) {
                uint32_t a[TB][16];
#pragma unroll
                for (int i = 0; i < TB; ++i) tmem_ld16(a[i], taddr + 16 * (b0 + i));
                tmem_wait_ld_boxes<TB>(a);
#pragma unroll
                for (int i = 0; i < TB; ++i) mma_box<KB, NH, F8>(acc, a[i], bf, b0 + i);
              }
            }
          } else {
#pragma unroll
            for (int s = 0; s < 4; ++s)
#pragma unroll
              for (int h = 0; h < NH; ++h)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[s][h][q] = 0.f;
          }
        } else if (tier == kTierStream) {
          // boxes in flight per batch: all of them when registers allow (one batch half, no register group),
          // two with both batch halves live, one in warps that also hold a register-resident group
          const int64_t v0 = row_base + (int64_t)kGroupRows * j + g;
          constexpr int SB = RFW ? 1 : ((NH == 1 || KB < 4) ? KB : 2);
#pragma unroll
          for (int b0 = 0; b0 < KB; b0 += SB) {
            uint32_t a[SB][16];
#pragma unroll
            for (int i = 0; i < SB; ++i) load_box_global_frag(a[i], P.W, v0, V, P.rw, b0 + i, c);
#pragma unroll
            for (int i = 0; i < SB; ++i) mma_box<KB, NH, F8>(acc, a[i], bf, b0 + i);
          }
        } else {
          if constexpr (RFW) {
#pragma unroll
            for (int bx = 0; bx < KB; ++bx) mma_box<KB, NH, F8>(acc, rfA[bx], bf, bx);
          } else {
#pragma unroll
            for (int s = 0; s < 4; ++s)
#pragma unroll
              for (int h = 0; h < NH; ++h)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[s][h][q] = 0.f;
          }
        }

        // z = p + base: each (row, walk) of the group belongs to one lane, which adds its projection to
        // the staged base logit in place (Fig. 7: projection summed, then added to the base logits)
        const int lr0 = kGroupRows * j + g;
        if constexpr (F8) {
          // E4M3 weights: columns 2c and 2c + 1 hold walk c's sums over its hi and lo vectors;
          // p = s_w (s1 sum_hi + s2 sum_lo)
          if (c < B) {
            const float h0 = __fadd_rn(__fadd_rn(acc[0][0][0], acc[1][0][0]), __fadd_rn(acc[2][0][0], acc[3][0][0]));
            const float l0 = __fadd_rn(__fadd_rn(acc[0][0][1], acc[1][0][1]), __fadd_rn(acc[2][0][1], acc[3][0][1]));
            const float h1 = __fadd_rn(__fadd_rn(acc[0][0][2], acc[1][0][2]), __fadd_rn(acc[2][0][2], acc[3][0][2]));
            const float l1 = __fadd_rn(__fadd_rn(acc[0][0][3], acc[1][0][3]), __fadd_rn(acc[2][0][3], acc[3][0][3]));
            const float p0 = __fmul_rn(s_sw[lr0], __fadd_rn(__fmul_rn(es1, h0), __fmul_rn(es2, l0)));
            const float p1 = __fmul_rn(s_sw[lr0 + 8], __fadd_rn(__fmul_rn(es1, h1), __fmul_rn(es2, l1)));
            float* zr = s_base + c * rows_cta + lr0;
            if constexpr (NB1) {
              zr[0] = __fadd_rn(p0, zb0);
              zr[8] = __fadd_rn(p1, zb1);
            } else {
              zr[0] = __fadd_rn(p0, zr[0]);
              zr[8] = __fadd_rn(p1, zr[8]);
            }
          }
        } else if constexpr (NB1) {
          if (c == 0) {
            s_base[lr0] = __fadd_rn(__fadd_rn(__fadd_rn(acc[0][0][0], acc[1][0][0]), __fadd_rn(acc[2][0][0], acc[3][0][0])),
                                    zb0);
            s_base[lr0 + 8] =
                __fadd_rn(__fadd_rn(__fadd_rn(acc[0][0][2], acc[1][0][2]), __fadd_rn(acc[2][0][2], acc[3][0][2])), zb1);
          }
        } else {
#pragma unroll
          for (int h = 0; h < NH; ++h)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int n = 8 * h + 2 * c + (q & 1);
              if (n < B) {
                const int idx = n * rows_cta + lr0 + ((q >> 1) << 3);
                s_base[idx] = __fadd_rn(
                    __fadd_rn(__fadd_rn(acc[0][h][q], acc[1][h][q]), __fadd_rn(acc[2][h][q], acc[3][h][q])), s_base[idx]);
              }
            }
        }
      }
      __syncthreads();

      // selection scan (Fig. 8, step 1): every thread scores rows of the CTA for one walk n = tid % Bp,
      // emits the logits (coalesced) and keeps the largest packed key
      if constexpr (NB1) {
        const int valid = (int)min((int64_t)rows_cta, V - row_base);
        const int64_t obase = (int64_t)t * V + row_base;
        unsigned long long bestk = 0ull;
        if (!sampled && !P.logits) {
          // greedy without logits: keys only (a loop of its own, so it carries no sampling code)
#pragma unroll 4
          for (int lr = tid; lr < valid; lr += kThreads)
            bestk = umax64(bestk, pack_key(s_base[lr], (uint32_t)(vg_base + lr)));
        } else if (!sampled) {
          for (int lr = tid; lr < valid; lr += kThreads) {
            const float z = s_base[lr];
            if (want_f32) reinterpret_cast<float*>(P.logits)[obase + lr] = z;
            else reinterpret_cast<__nv_bfloat16*>(P.logits)[obase + lr] = __float2bfloat16_rn(z);
            bestk = umax64(bestk, pack_key(z, (uint32_t)(vg_base + lr)));
          }
        } else {
          // sampled: each thread scores four consecutive rows with one Philox call (the CTA's first row is a
          // multiple of 16, and so is the shard's first row: vg_base + lr is a multiple of 4)
          for (int lr = 4 * tid; lr < valid; lr += 4 * kThreads) {
            const float4 z4 = *reinterpret_cast<const float4*>(s_base + lr);
            const float zz[4] = {z4.x, z4.y, z4.z, z4.w};
            const uint32_t v0 = (uint32_t)(vg_base + lr);
            const uint4 o = philox_quad(P.seed, 0u, tau, v0 >> 2);
            const uint32_t ww[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (lr + u < valid) {
                if (P.logits) {
                  if (want_f32) reinterpret_cast<float*>(P.logits)[obase + lr + u] = zz[u];
                  else reinterpret_cast<__nv_bfloat16*>(P.logits)[obase + lr + u] = __float2bfloat16_rn(zz[u]);
                }
                const float key = __fadd_rn(t_is_one ? zz[u] : __fdiv_rn(zz[u], T), gumbel_from_word(ww[u]));
                bestk = umax64(bestk, pack_key(key, v0 + (uint32_t)u));
              }
            }
          }
        }
        const unsigned long long wk = warp_max64((uint32_t)(bestk >> 32), (uint32_t)bestk);
        if (lane == 0) s_red[warp * kMaxB] = wk;
      } else {
        const int Bp = B == 1 ? 1 : B == 2 ? 2 : B <= 4 ? 4 : B <= 8 ? 8 : 16;
        const int n = tid & (Bp - 1);
        const int stride = kThreads / Bp;
        unsigned long long bestk = 0ull;
        if (n < B) {
          const float* zrow = s_base + n * rows_cta;
          const int valid = (int)min((int64_t)rows_cta, V - row_base);
          const int64_t obase = ((int64_t)n * gamma + t) * V + row_base;
          if (!sampled && !P.logits) {
#pragma unroll 4
            for (int lr = tid / Bp; lr < valid; lr += stride)
              bestk = umax64(bestk, pack_key(zrow[lr], (uint32_t)(vg_base + lr)));
          } else if (!sampled) {
            for (int lr = tid / Bp; lr < valid; lr += stride) {
              const float z = zrow[lr];
              if (want_f32) reinterpret_cast<float*>(P.logits)[obase + lr] = z;
              else reinterpret_cast<__nv_bfloat16*>(P.logits)[obase + lr] = __float2bfloat16_rn(z);
              bestk = umax64(bestk, pack_key(z, (uint32_t)(vg_base + lr)));
            }
          } else {
            // sampled: four consecutive rows per Philox call, as for a single walk
            for (int lr = 4 * (tid / Bp); lr < valid; lr += 4 * stride) {
              const float4 z4 = *reinterpret_cast<const float4*>(zrow + lr);
              const float zz[4] = {z4.x, z4.y, z4.z, z4.w};
              const uint32_t v0 = (uint32_t)(vg_base + lr);
              const uint4 o = philox_quad(P.seed, (uint32_t)n, tau, v0 >> 2);
              const uint32_t ww[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                if (lr + u < valid) {
                  if (P.logits) {
                    if (want_f32) reinterpret_cast<float*>(P.logits)[obase + lr + u] = zz[u];
                    else reinterpret_cast<__nv_bfloat16*>(P.logits)[obase + lr + u] = __float2bfloat16_rn(zz[u]);
                  }
                  const float key = __fadd_rn(t_is_one ? zz[u] : __fdiv_rn(zz[u], T), gumbel_from_word(ww[u]));
                  bestk = umax64(bestk, pack_key(key, v0 + (uint32_t)u));
                }
              }
            }
          }
        }
        for (int off = 16; off >= Bp; off >>= 1) bestk = umax64(bestk, __shfl_xor_sync(0xffffffffu, bestk, off));
        if (lane < Bp && n < B) s_red[warp * kMaxB + n] = bestk;
      }

      __syncthreads();
      trace_stamp(P, 2 + kTraceStampsPerStep * t + 1);

      // the other warps fetch the next step's base logits while warp 0 runs the exchange; with asynchronous
      // copies each thread takes the rows it had copied a step earlier and starts the copy for the step after
      if constexpr (base_async) {
        if (tid >= 32) {
          asm volatile("cp.async.wait_all;" ::: "memory");
          move_base(P, s_base, s_base_in, t + 1, 32, kThreads - 32);
          copy_base_async(P, s_base_in, row_base, t + 2, 32, kThreads - 32);
        }
      } else if constexpr (NB1) {
        stage_base(P, s_base, row_base, t + 1, 32, kThreads - 32);
      } else {
        // several walks: a few rows per walk and thread, so the copies run asynchronously (measured faster than
        // register loads from B = 2 up; slower for one walk)
        stage_base_cp(P, s_base, row_base, t + 1, 32, kThreads - 32);
      }

      // exchange (Fig. 8). Each CTA publishes its winner for walk n as one 64-bit word in its own slot,
      // tag (step + 1) << 56 | ord(key) << 24 | (2^24 - 1 - row), with a relaxed store: an aligned 64-bit store
      // is single-copy atomic, so a reader sees the old word or the new one and the tag says which. A relaxed
      // arrival count tells the readers when to look; a reader re-reads any slot whose tag is not yet this
      // step's. No fence is needed because the answer is taken only from words that carry this step's tag.
      // Slots alternate between two step buffers: a CTA can reach step t + 2 only after every CTA has
      // arrived at step t + 1, that is, after every CTA has finished reading step t's buffer. A buffer is
      // walk-major (walk n's slots of all CTAs side by side), so reading one walk's slots touches G / 16
      // lines rather than one line per CTA (measured: 16 walks, gamma = 16, 288 -> 243 us per walk).
      if (!RFW && warp == 0) {
        unsigned long long kk = 0ull;
        if constexpr (NB1) {
          // one walk: lane w reads warp w's key, and the warp maximum goes to every lane
          const unsigned long long mine = (lane < kWarps) ? s_red[lane * kMaxB] : 0ull;
          kk = warp_max64((uint32_t)(mine >> 32), (uint32_t)mine);
        } else {
          if (lane < B)
            for (int w = 0; w < kWarps; ++w) kk = umax64(kk, s_red[w * kMaxB + lane]);
        }
        unsigned long long* sl = P.slots + (int64_t)(t & 1) * G * B;
        const unsigned long long tag = (unsigned long long)(t + 1) << 56;
        const bool skip = (P.flags & kFlagSkipArrival) && cta == 0 && t == 0;
        if (lane < B && !skip) {
          unsigned long long k56 = 0ull;
          if (kk != 0ull) {
            const uint32_t v = 0xFFFFFFFFu - (uint32_t)(kk & 0xFFFFFFFFull);
            k56 = ((kk >> 32) << 24) | (unsigned long long)(0xFFFFFFu - v);
          }
          asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(sl + (int64_t)lane * G + cta), "l"(tag | k56) : "memory");
        }
        __syncwarp();
        const uint64_t t_start = globaltimer_ns();
        if (lane == 0 && !skip) asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(P.cnt) : "memory");
        // the E row of this CTA's candidate goes to L2 while the others arrive: if it wins, every CTA reads it
        // right after the wait (issued after the arrival so that it cannot hold the arrival back)
        if (lane < B && kk != 0ull && !(P.flags & kFlagFixedLatent)) {
          const uint16_t* er = P.E + (int64_t)(0xFFFFFFFFu - (uint32_t)(kk & 0xFFFFFFFFull)) * r;
          for (int off = 0; off < r * 2; off += 128) prefetch_l2(reinterpret_cast<const uint8_t*>(er) + off);
        }
        // The counter only says when to look: once all but 64 CTAs have arrived (measured: 96.5 us per walk against
        // 98.4 when waiting for all but 4; reading every slot from the start was no better), every poll also reads the
        // slots, and the step is complete exactly when every slot carries this step's tag.
        constexpr int kSlotsPerLane = kMaxGrid / 32;
        const unsigned int target = (unsigned int)(t + 1) * (unsigned int)G;
        const unsigned int near = target - (unsigned int)min(G, 64);
        bool late = false;
        if constexpr (kParRead) {
          // several walks: this warp waits only until all but 64 CTAs have arrived; after the barrier below
          // the warps read the slots of their walks side by side
          for (uint32_t spins = 0;; ) {
            unsigned int now = 0;
            if (lane == 0) asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(now) : "l"(P.cnt) : "memory");
            if (__shfl_sync(0xffffffffu, now, 0) >= near) break;
            if ((++spins & 15u) == 0u && __any_sync(0xffffffffu, globaltimer_ns() - t_start > P.timeout_ns)) {
              late = true;
              break;
            }
          }
        }
        for (int n = 0; n < B && !late && !kParRead; ++n) {
          unsigned long long w[kSlotsPerLane];
#pragma unroll
          for (int i = 0; i < kSlotsPerLane; ++i) w[i] = (lane + 32 * i < G) ? 0ull : tag;  // tag 0: not read yet
          uint32_t spins = 0;
          bool counted = (n > 0);  // later walks: everyone has arrived already
          while (true) {
            if (!counted) {
              unsigned int now = 0;
              if (lane == 0) asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(now) : "l"(P.cnt) : "memory");
              now = __shfl_sync(0xffffffffu, now, 0);
              counted = now >= near;
            }
            bool fresh = true;
            if (counted) {
#pragma unroll
              for (int i = 0; i < kSlotsPerLane; ++i) {
                const int cc = lane + 32 * i;
                if (cc < G && (w[i] >> 56) != (unsigned long long)(t + 1))
                  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w[i]) : "l"(sl + (int64_t)n * G + cc) : "memory");
              }
#pragma unroll
              for (int i = 0; i < kSlotsPerLane; ++i) fresh = fresh && ((w[i] >> 56) == (unsigned long long)(t + 1));
            }
            if (__all_sync(0xffffffffu, counted && fresh)) break;
            // the time-out decision is made by the whole warp at once, so the lanes leave the loop together
            if ((++spins & 15u) == 0u && __any_sync(0xffffffffu, globaltimer_ns() - t_start > P.timeout_ns)) {
              late = true;
              break;
            }
          }
          late = __any_sync(0xffffffffu, late);
          if (late) break;
          unsigned long long best = 0ull;
#pragma unroll
          for (int i = 0; i < kSlotsPerLane; ++i) best = umax64(best, w[i] & 0x00FFFFFFFFFFFFFFull);
          const unsigned long long wk = warp_max64((uint32_t)(best >> 32), (uint32_t)best);
          if (lane == 0) {
            const int32_t x = (int32_t)(0xFFFFFFu - ((uint32_t)wk & 0xFFFFFFu));
            s_win[n] = x;
            if (cta == 0) {
              P.tokens[(int64_t)n * gamma + t] = x;
              if (P.keys) P.keys[(int64_t)n * gamma + t] = ((wk >> 24) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)x);
            }
          }
        }
        late = __any_sync(0xffffffffu, late);
        if (late && lane == 0) {
          atomicCAS(P.status, 0, kStatusTimeout);
          *s_abort = 1;
        }
        // E4M3 weights, Markov, one walk: the winner's E row, split into two E4M3 vectors, for every warp's next
        // B fragments (a winner outside W is skipped here; the check after the barrier ends the walk)
        if constexpr (F8 && !kParRead) {
          if (!late && !recurrent && !(P.flags & kFlagFixedLatent)) {
            __syncwarp();
            split_winner_rows();
          }
        }
        if constexpr (!kParRead) trace_stamp(P, 2 + kTraceStampsPerStep * t + 2);
      }
      if constexpr (kParRead) {
        // several walks: every warp that keeps no register group reads the slots of walks k, k + m, ...
        // (k its rank among those m warps), so the walks' reads overlap instead of following one another
        __syncthreads();
        if constexpr (!RFW) {
          if (!*s_abort) {
            const uint32_t others = ~P.rf_warp_mask & ((1u << kWarps) - 1u);
            const int m = __popc(others), k = __popc(others & ((1u << warp) - 1u));
            const unsigned long long* sl = P.slots + (int64_t)(t & 1) * G * B;
            const uint64_t t_w = globaltimer_ns();
            bool late = false;
            for (int n = k; n < B; n += m) {
              const unsigned long long wk = read_walk_slots<kMaxGrid / 32>(sl, G, B, n, t, lane, t_w, P.timeout_ns, late);
              if (late) break;
              if (lane == 0) {
                const int32_t x = (int32_t)(0xFFFFFFu - ((uint32_t)wk & 0xFFFFFFu));
                s_win[n] = x;
                if (cta == 0) {
                  P.tokens[(int64_t)n * gamma + t] = x;
                  if (P.keys)
                    P.keys[(int64_t)n * gamma + t] = ((wk >> 24) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)x);
                }
              }
            }
            if (late && lane == 0) {
              atomicCAS(P.status, 0, kStatusTimeout);
              *s_abort = 1;
            }
          }
        }
        trace_stamp(P, 2 + kTraceStampsPerStep * t + 2);
      }
      // the next step's base logits have landed in shared memory before the barrier
      if constexpr (!base_async && !NB1) asm volatile("cp.async.wait_all;" ::: "memory");
      __syncthreads();
      if (*s_abort) break;

      // winners must be rows of W (a failed exchange would show up here)
      bool bad = false;
      for (int n = 0; n < B; ++n) bad |= ((int64_t)s_win[n] < P.v_offset || (int64_t)s_win[n] >= P.v_offset + V);
      if (bad) {
        if (tid == 0) atomicCAS(P.status, 0, kStatusInternal);
        break;
      }

      // ---------------- state advance ----------------
      if (P.flags & kFlagFixedLatent) continue;
      // after the last step the state is needed only when the caller asks for the states
      if (t + 1 == gamma && P.state == nullptr) {
        trace_stamp(P, 2 + kTraceStampsPerStep * t + 3);
        break;
      }
      if (!recurrent) {
        if constexpr (F8) {
          if constexpr (kParRead) {
            // several walks: the winners are known only after the barrier, so warp 0 splits their E rows now
            if constexpr (!RFW) {
              if (warp == 0) split_winner_rows();
            }
            __syncthreads();
          }
          // the winners' E rows are split in shared memory
          bfrag_from_split_smem<KB>(bf, es1, es2, s_q, s_qs, B, r, lane);
        } else {
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const int n = 8 * h + g;
            if (n < B) bfrag_from_bf16_row<KB>(bf[h], P.E + (int64_t)s_win[n] * r, c);
          }
        }
        if (cta == 0 && P.state) {
          for (int i = tid; i < B * r; i += kThreads) {
            const int n = i / r, k = i % r;
            const uint32_t bits = (uint32_t)P.E[(int64_t)s_win[n] * r + k] << 16;
            P.state[((int64_t)n * gamma + t) * r + k] = __uint_as_float(bits);
          }
        }
      } else {
        // the slices carry step t's tag once their stores are visible (every CTA wrote its slice before it
        // arrived, so the wait is short); running out of time sets the time-out status and ends the walk
        const unsigned long long* ah = P.ah + (int64_t)(t & 1) * B * r;
        const uint64_t t_wait = globaltimer_ns();
        bool ah_late = false;
        for (int i = tid; i < B * r; i += kThreads) {
          const int n = i / r, k = i % r;
          const float e = __uint_as_float((uint32_t)P.E[(int64_t)s_win[n] * r + k] << 16);
          const float ck = P.c ? P.c[k] : 0.f;  // loaded beside E's row, ahead of the slice reads
          unsigned long long word = 0ull;
          for (uint32_t spins = 0;; ++spins) {
            asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(word) : "l"(ah + i) : "memory");
            if ((uint32_t)(word >> 32) == (uint32_t)(t + 1)) break;
            if ((spins & 15u) == 15u && globaltimer_ns() - t_wait > P.timeout_ns) {
              ah_late = true;
              break;
            }
          }
          if (ah_late) break;
          float pre = __fadd_rn(__uint_as_float((uint32_t)word), e);
          if (P.c) pre = __fadd_rn(pre, ck);
          s_h[i] = tanhf(pre);
        }
        if (ah_late) {
          atomicCAS(P.status, 0, kStatusTimeout);
          *s_abort = 1;
        }
        __syncthreads();
        if constexpr (F8) {
          if (warp == 0)
            split_state_smem<KB>(s_q, s_qs, B, r, lane, [&](int w, auto& x) {
              const float* src = s_h + w * r + lane * 4 * KB;
#pragma unroll
              for (int e = 0; e < 4 * KB; ++e) x[e] = src[e];
            });
          __syncthreads();
          bfrag_from_split_smem<KB>(bf, es1, es2, s_q, s_qs, B, r, lane);
        } else {
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const int n = 8 * h + g;
            if (n < B) bfrag_from_f32<KB>(bf[h], s_h + n * r, c);
          }
        }
        if (cta == 0 && P.state) {
          for (int i = tid; i < B * r; i += kThreads) {
            const int n = i / r, k = i % r;
            P.state[((int64_t)n * gamma + t) * r + k] = s_h[i];
          }
        }
      }
      trace_stamp(P, 2 + kTraceStampsPerStep * t + 3);
    }
  };
  if (rf_warp) walk(std::true_type{});
  else walk(std::false_type{});

  // ---------------- exit ----------------
  // copies still in flight after a timed-out wait must land before the CTA's shared memory is released
  if (!tma_done) (void)mbar_wait_bounded(mbar, 0u, P.timeout_ns);
  asm volatile("cp.async.wait_all;" ::: "memory");
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  if (warp == 0 && P.tmem_cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(P.tmem_cols) : "memory");
  }
}

}  // namespace whead
