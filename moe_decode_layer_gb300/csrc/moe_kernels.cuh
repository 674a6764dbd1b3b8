// Kernels of the small-batch MoE decode layer step (sm_103a).
//
// Every CTA has kNC consumer warps and one producer warp. The producer streams
// weights from HBM into a ring of shared-memory slots with 1-D bulk (TMA)
// copies tagged evict-first in L2. A stage is a block of consecutive rows
// (several router row pairs, several gate/up row pairs of one expert as one
// gate block and one up block, or one expert's down rows for this CTA's output
// features), so each stage needs few large copies: the copy engine's rate per SM
// is bounded by copies and stages issued, not by bytes in flight. Each slot has
// a "full" mbarrier (the copy engine counts the bytes in) and an "empty"
// mbarrier (the consumers hand the slot back).
//
// Phases (Ling-3.0-flash batch-1 decode blog, section "PDL: stacking the latency
// floors of small kernels": router chain norm -> gate matvec -> top-k, MoE chain
// up-GEMM -> activation -> down-GEMM -> combine):
//   R  router rows (bf16) and the shared experts' gate/up rows: router logits and
//      the shared experts' silu(g) * u; neither needs a routing decision.
//   T  every CTA reads all logits and selects the top-k of each row itself, then
//      forms the union of chosen experts from one row mask per expert and counts
//      of the chosen ids below each expert (SGLang Low-Latency Mode page, section
//      "Low-Latency-Specific Optimizations", item 3: with at most eight rows the
//      experts are placed by row masks and population counts, not by a sort).
//   U  gate/up rows of the chosen experts: h = w * silu(g) * u per (expert, row),
//      SwiGLU in fp32 right after the dot products (blog section "Two fusions and
//      a retune"). Row pairs of a stage go to different consumer warps.
//   D  down rows: each CTA owns a contiguous block of output features, sums
//      W2_e h_e over all chosen and shared experts in fp32 and writes
//      bf16(residual + sum) with one rounding (blog section "PDL: ...": the combine
//      is an fp32 sum with a single final cast).
//
// Router logits pass between CTAs without a fence or a flag: every value is a
// 64-bit word (run tag << 32 | fp32 bits) and readers poll until the tag equals
// the current run's tag ("Muse Spark Open Ultrafast", section "Megakernel
// internals", part 3: a GPU-scope fence with bulk loads in flight costs
// microseconds, so the data carries its own readiness). The tag is a per-handle
// counter that the last CTA of a run advances, so buffers are never reset. The
// h values (I floats per (expert, row) pair, in pair order, four copies) go
// through global memory too:
//   - moe_layer_kernel (phases in order, and the three-kernel chain): each CTA
//     releases its h once by a fence and a count; after the count reaches the
//     grid size each CTA fetches its batches of pairs with one bulk copy each,
//     the next batch landing while the current one is in use.
//   - moe_ilv_kernel (slot-interleaved): each CTA computes a block of rows of
//     every union slot; per slot, a hand-off warp fences once and counts the
//     CTA's items, and another copies the slot's h rows behind the down weights
//     of that slot's down stage once every CTA has counted it. The down stage of
//     slot s follows the gate/up items of slot s + lag, so gate/up and down
//     weights stream as one sequence and no CTA waits for all gate/up results.
//
// All device functions are inlined into the kernel: parameters are then read
// from the kernel's parameter space and the helper objects stay in registers
// (through a reference in a separate function both would be memory loads).
//
// Every wait (mbarrier, tagged poll) is bounded by the handle's wait limit; on
// expiry the CTA records DEV_ERR_TIMEOUT in the status word, stops issuing
// copies, skips the arithmetic, keeps every barrier of the schedule, drains its
// own bulk copies and exits.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "moe_params.h"
#include "ptx.cuh"

namespace moe {

constexpr uint32_t kFull = 0xffffffffu;
constexpr int kBarConsumers = 1;  // named barrier: the kNC consumer warps
constexpr int kBarRoute = 2;      // named barrier: consumers -> producer, routing ready
constexpr int kBarRouting = 3;    // named barrier: the routing warps (single-kernel schedules)
constexpr int kStageBatch = 8;    // tagged words in flight per thread when staging h

// --------------------------------------------------------------------------
// small helpers
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// [lo, hi) share of n items for CTA c of g (n * g < 2^32 for every phase).
__device__ __forceinline__ void split_range(int n, int c, int g, int& lo, int& hi) {
  lo = (int)((unsigned)n * (unsigned)c / (unsigned)g);
  hi = (int)((unsigned)n * (unsigned)(c + 1) / (unsigned)g);
}

// Slot-interleaved schedule: the gate/up rows [lo, hi) of union slot s that
// this CTA computes. Each slot's I rows are split over all CTAs; the map from
// CTA to row block rotates from slot to slot, so the CTAs given one row more
// differ between slots.
__device__ __forceinline__ void ilv_rows(const Params& p, int s, int& lo, int& hi) {
  const int c = (int)((blockIdx.x + (unsigned)s * (unsigned)kIlvRot) % (unsigned)p.grid);
  split_range(p.I, c, p.grid, lo, hi);
}
// Interleaved schedule: consumer warps 0 .. ilv_nrw - 1 route; the others
// compute the shared experts' gate/up items meanwhile, in stages of at most
// ilv_sq pairs (one item per warp and stage).
__device__ __forceinline__ int ilv_nrw(const Params& p) { return max(p.M, 2); }
// warps that compute the shared experts' items while the routing runs
__device__ __forceinline__ int ilv_snw(const Params& p) { return kNC - ilv_nrw(p); }
__device__ __forceinline__ int ilv_sq(const Params& p) { return min(p.q, ilv_snw(p)); }
// Threads meeting at the routing-ready barrier: the routing warps, the producer
// and the two hand-off warps.
__device__ __forceinline__ int ilv_route_threads(const Params& p) { return (ilv_nrw(p) + 3) * 32; }

// Position in the shared-memory ring: stage number, its slot and the slot's
// mbarrier phase parity, advanced without divisions.
// The slot count may differ between phases (the routed gate/up stages also use
// the extra slots), so each slot keeps its own use parity.
struct Ring {
  int seq = 0, slot = 0;
  uint64_t par = 0;  // bit s: parity of slot s's current use
  __device__ __forceinline__ uint32_t phase() const { return (uint32_t)(par >> slot) & 1u; }
  __device__ __forceinline__ void next(int nslots) {
    ++seq;
    par ^= 1ull << slot;
    if (++slot >= nslots) slot = 0;
  }
  // Entering a phase with fewer slots: the next stage must be one of them.
  __device__ __forceinline__ void fit(int nslots) {
    if (slot >= nslots) slot = 0;
  }
};

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

struct Ctx {
  const Params& p;
  uint8_t* sm;
  int* misc;
  volatile int* slot_seq;  // [nslots] ring stage that currently owns each slot
  uint32_t full0, empty0, xbar;
  uint64_t t0;
  long long c0;
  int tid, warp, lane;

  __device__ __forceinline__ Ctx(const Params& pp, uint8_t* base) : p(pp), sm(base) {
    misc = reinterpret_cast<int*>(sm + p.off_misc);
    slot_seq = reinterpret_cast<volatile int*>(sm + p.off_slot_seq);
    full0 = smem_u32(sm + p.off_full);
    empty0 = smem_u32(sm + p.off_empty);
    xbar = smem_u32(sm + p.off_xbar);
    t0 = global_ns();
    c0 = clock64();
    tid = threadIdx.x;
    warp = tid >> 5;
    lane = tid & 31;
  }
  __device__ __forceinline__ bool aborted() const { return *reinterpret_cast<volatile int*>(misc + MISC_ABORT) != 0; }
  __device__ __forceinline__ void fail(uint32_t site) const {
    *reinterpret_cast<volatile int*>(misc + MISC_ABORT) = 1;
    atomicOr(&p.ctrl[CTRL_STATUS], DEV_ERR_TIMEOUT);
    atomicCAS(&p.ctrl[CTRL_WHERE], 0u, site);
  }
  // Stop this CTA's waits without a status of its own (another CTA set one).
  __device__ __forceinline__ void abort_local() const { *reinterpret_cast<volatile int*>(misc + MISC_ABORT) = 1; }
  __device__ __forceinline__ bool expired() const { return global_ns() - t0 > p.timeout_ns; }
  // Another CTA gave up: stop waiting on data it will never publish.
  __device__ __forceinline__ bool peer_failed() const { return ld_relaxed_u32(&p.ctrl[CTRL_STATUS]) != 0; }
  __device__ __forceinline__ uint32_t epoch() const { return static_cast<uint32_t>(misc[MISC_EPOCH]); }
  // Slots past nslots: in the gate/up phase extra slots in the h area, in the
  // down phase (d) the x area.
  __device__ __forceinline__ uint8_t* slot_ptr(int slot, bool d = false) const {
    return slot < p.nslots ? sm + p.off_ring + (size_t)slot * p.slot_bytes
           : d             ? sm + p.off_x
                           : sm + p.off_xslot + (size_t)(slot - p.nslots) * p.slot_bytes;
  }
  // Phase timestamp (one plain store; off unless the handle has a stamp buffer).
  __device__ __forceinline__ void stamp(int ev) const {
    if (p.stamps) p.stamps[(size_t)blockIdx.x * kStampSlots + ev] = global_ns();
  }
  __device__ __forceinline__ void count(int ev, unsigned long long v) const {
    if (p.stamps) atomicAdd(&p.stamps[(size_t)blockIdx.x * kStampSlots + ev], v);
  }

  // Bounded wait on an mbarrier phase. False on abort / timeout.
  __device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t par, uint32_t site) const {
    while (!mbar_try_wait(bar, par)) {
      if (aborted()) return false;
      if (expired()) {
        fail(site);
        return false;
      }
    }
    return true;
  }

  // Bounded wait for ring stage `seq` to be full. Consumer warps take stages
  // out of step with each other, so a warp may ask for a stage more than one lap
  // ahead of its slot; an mbarrier parity only tells adjacent phases apart. The
  // producer therefore records which stage owns a slot before arming it, and the
  // parity wait starts only once `seq` owns the slot.
  __device__ __forceinline__ bool wait_full(const Ring& r) const {
    for (uint32_t spin = 0; slot_seq[r.slot] != r.seq; ++spin) {
      __nanosleep(64);  // leave the issue slots to the warps doing arithmetic
      if ((spin & 15) == 15) {
        if (aborted()) return false;
        if (expired()) {
          fail(SITE_RING_FULL);
          return false;
        }
      }
    }
    return wait_bar(full0 + 8u * r.slot, r.phase(), SITE_RING_FULL);
  }
  // Producer side: bounded wait for the slot of stage `r` to be free.
  __device__ __forceinline__ bool wait_empty(const Ring& r) const {
    return wait_bar(empty0 + 8u * r.slot, r.phase() ^ 1u, SITE_RING_EMPTY);
  }
  __device__ __forceinline__ void release(const Ring& r, uint32_t count) const { mbar_arrive(empty0 + 8u * r.slot, count); }
};

// Routing tables in shared memory.
struct Route {
  int* sel_e;           // [maxm][K] chosen experts, descending weight
  float* sel_w;         // [maxm][K]
  uint32_t* emask;      // [E] row mask per expert
  uint32_t* bitmap;     // [E / 32] experts chosen by any row
  int* slot_of;         // [E] union slot of a chosen expert
  int* slot_e;          // [nslot_max] expert id, or -1 - s for shared expert s
  uint32_t* slot_mask;  // [nslot_max] rows that use the slot
  float* slot_w;        // [nslot_max][maxm] combine weight (routed_scale folded in)
  int* pair_base;       // [nslot_max + 1] first (slot, row) pair index of each slot
  __device__ __forceinline__ Route(const Params& p, uint8_t* sm)
      : sel_e(reinterpret_cast<int*>(sm + p.off_sel_e)),
        sel_w(reinterpret_cast<float*>(sm + p.off_sel_w)),
        emask(reinterpret_cast<uint32_t*>(sm + p.off_emask)),
        bitmap(reinterpret_cast<uint32_t*>(sm + p.off_bitmap)),
        slot_of(reinterpret_cast<int*>(sm + p.off_slot_of)),
        slot_e(reinterpret_cast<int*>(sm + p.off_slot_e)),
        slot_mask(reinterpret_cast<uint32_t*>(sm + p.off_slot_mask)),
        slot_w(reinterpret_cast<float*>(sm + p.off_slot_w)),
        pair_base(reinterpret_cast<int*>(sm + p.off_pair_base)) {}
};

// Hand-off counters: after storing its share of a phase's results, every CTA
// adds one to a 64-bit counter; readers wait (one thread per CTA, bounded, with
// back-off) until it reaches the grid size. The count is only a cheap readiness
// hint -- one word polled per CTA instead of every result -- and the results are
// still read with their own tag check. The last CTA of a run resets the counters.
__device__ __forceinline__ void count_done(const Params& p, int word) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], 1;" ::"l"(p.ctrl + word) : "memory");
}
static __device__ __forceinline__ bool wait_count(const Ctx& c, int word, uint32_t site) {
  const Params& p = c.p;
  const unsigned long long* cnt = reinterpret_cast<const unsigned long long*>(p.ctrl + word);
  for (uint32_t spin = 0; ld_relaxed_u64(cnt) < (unsigned long long)p.grid; ++spin) {
    __nanosleep(100);
    if ((spin & 15) == 15) {
      if (c.aborted() || c.peer_failed()) return false;
      if (c.expired()) {
        c.fail(site);
        return false;
      }
    }
  }
  return true;
}

// --------------------------------------------------------------------------
// stage schedule: the same walk on the producer and the consumer side
// --------------------------------------------------------------------------
// Items of the gate/up phases are (slot u, row j) pairs flattened as u * I + j;
// a stage holds up to q consecutive items of one slot (expert). Router items are
// row pairs; a stage holds up to qr of them (no slot boundaries). Item t of the
// CTA's range [lo, hi) goes to consumer warp (t - lo) % kNC.
struct ItemWalk {
  int a, hi, u, j, r;  // next item, end, its slot and row, (a - lo) % nw
  int q, I;            // items per stage, rows per slot (0: no boundaries)
  int w0 = 0, nw = kNC;  // the warps that take items: w0 .. w0 + nw - 1 (q <= nw)
  __device__ __forceinline__ ItemWalk(int lo, int hi_, int q_, int I_) : a(lo), hi(hi_), r(0), q(q_), I(I_) {
    u = I_ > 0 ? lo / I_ : 0;
    j = I_ > 0 ? lo - u * I_ : lo;
  }
  __device__ __forceinline__ bool more() const { return a < hi; }
  // items in the current stage
  __device__ __forceinline__ int count() const {
    int n = min(q, hi - a);
    if (I > 0) n = min(n, I - j);
    return n;
  }
  // offset of warp w's item in the current stage (>= count() when it has none)
  __device__ __forceinline__ int offset(int w) const {
    if (w < w0 || w >= w0 + nw) return kNC;
    const int d = w - w0 - r;
    return d < 0 ? d + nw : d;
  }
  __device__ __forceinline__ void advance(int n) {
    a += n;
    j += n;
    if (I > 0 && j == I) {
      j = 0;
      ++u;
    }
    r += n;
    if (r >= nw) r -= nw;
  }
};

// --------------------------------------------------------------------------
// consumer: x rows (arrive by bulk copy; optionally RMS-normalised in place)
// --------------------------------------------------------------------------
// row_max (NVFP4 / FP8 weights): also each row's largest |x| as bf16 bits into
// MISC_XMAX + m (one warp per row, after the normalisation), while the router
// stages are still landing; x_to_f16 scales by it after routing.
static __device__ __forceinline__ void prepare_x(const Ctx& c, bool row_max = false) {
  const Params& p = c.p;
  if (!c.wait_bar(c.xbar, 0, SITE_RING_FULL)) return;
  uint4* xs = reinterpret_cast<uint4*>(c.sm + p.off_x);
  const int nch = p.H / 8;
  if (p.pre_rmsnorm) {
    for (int m = c.warp; m < p.M; m += kNC) {
      float ss = 0.0f;
      for (int ch = c.lane; ch < nch; ch += 32) {
        const uint4 v = xs[m * nch + ch];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float a = bf16lo(w[q]), b = bf16hi(w[q]);
          ss = fmaf(a, a, ss);
          ss = fmaf(b, b, ss);
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
      const float scale = 1.0f / sqrtf(ss / (float)p.H + p.rms_eps);
      for (int ch = c.lane; ch < nch; ch += 32) {
        const uint4 v = xs[m * nch + ch];
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t lo = f32_to_bf16_bits(bf16lo(w[q]) * scale);
          const uint32_t hi = f32_to_bf16_bits(bf16hi(w[q]) * scale);
          w[q] = lo | (hi << 16);
        }
        xs[m * nch + ch] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  if (row_max) {
    __syncwarp();  // the warp's normalised rows before it reads them back
    uint32_t* xmax = reinterpret_cast<uint32_t*>(c.misc + MISC_XMAX);
    for (int m = c.warp; m < p.M; m += kNC) {
      uint32_t a = 0u;  // |x| as bits: larger bits, larger value
      for (int ch = c.lane; ch < nch; ch += 32) {
        const uint4 v = xs[m * nch + ch];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) a = max(a, max(w[q] & 0x7fffu, (w[q] >> 16) & 0x7fffu));
      }
      a = warp_max_u32(a);
      if (c.lane == 0) xmax[m] = a;
    }
  }
}

// --------------------------------------------------------------------------
// consumer: dot products of one row pair with the token rows in `mask`.
// Results are warp-reduced (butterfly), so every lane holds all sums.
// --------------------------------------------------------------------------
// Sums of one (gate row, up row) item for one x row, held by one lane after
// the warp reduction: lane k holds the k-th row of the item's row mask (m = -1
// on lanes without a row).
struct RowSums {
  int m;
  float g, u;
};

__device__ __forceinline__ void warp_sum2(float& g, float& u) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    g += __shfl_xor_sync(kFull, g, o);
    u += __shfl_xor_sync(kFull, u, o);
  }
}

// bf16 rows a, b against one x row held in the lane's registers (xr: chunks
// lane, lane + 32, ...). Two partial sums per row (even / odd chunk) shorten
// the dependent FMA chain.
__device__ __forceinline__ RowSums dot_one_bf16(const uint4* wa, const uint4* wb, int nch, const uint4* xr,
                                                int lane) {
  float g0 = 0.f, g1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
  for (int i = 0; i < kCplBf16; i += 2) {
    const int ch0 = lane + 32 * i, ch1 = ch0 + 32;
    if (ch0 < nch) {
      dot8_bf16(g0, wa[ch0], xr[i]);
      dot8_bf16(u0, wb[ch0], xr[i]);
    }
    if (ch1 < nch) {
      dot8_bf16(g1, wa[ch1], xr[i + 1]);
      dot8_bf16(u1, wb[ch1], xr[i + 1]);
    }
  }
  RowSums r{0, g0 + g1, u0 + u1};
  warp_sum2(r.g, r.u);
  if (lane != 0) r.m = -1;
  return r;
}

// bf16 rows a, b against the N x rows of `mask` (N = popcount), x rows in
// shared memory. Only the rows that chose the expert are computed; two chunks
// per step give each row four independent FMA chains.
template <int N>
__device__ __forceinline__ RowSums dot_rows_bf16(const uint4* wa, const uint4* wb, int nch, const uint4* xs,
                                                 uint32_t mask, int lane) {
  int rows[N];
  const uint4* xp[N];
  uint32_t msk = mask;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    rows[k] = __ffs(msk) - 1;
    msk &= msk - 1;
    xp[k] = xs + rows[k] * nch;
  }
  float g0[N], g1[N], u0[N], u1[N];
#pragma unroll
  for (int k = 0; k < N; ++k) g0[k] = g1[k] = u0[k] = u1[k] = 0.0f;
  int ch = lane;
  if (N <= 4) {  // two chunks per step while the registers allow it
    for (; ch + 32 < nch; ch += 64) {  // nch is a multiple of 32: the trip count is warp-uniform
      const uint4 a0 = wa[ch], b0 = wb[ch], a1 = wa[ch + 32], b1 = wb[ch + 32];
#pragma unroll
      for (int k = 0; k < N; ++k) {
        const uint4 x0 = xp[k][ch], x1 = xp[k][ch + 32];
        dot8_bf16(g0[k], a0, x0);
        dot8_bf16(u0[k], b0, x0);
        dot8_bf16(g1[k], a1, x1);
        dot8_bf16(u1[k], b1, x1);
      }
    }
  }
  for (; ch < nch; ch += 32) {
    const uint4 a0 = wa[ch], b0 = wb[ch];
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const uint4 x0 = xp[k][ch];
      dot8_bf16(g0[k], a0, x0);
      dot8_bf16(u0[k], b0, x0);
    }
  }
  RowSums r{-1, 0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < N; ++k) {
    float g = g0[k] + g1[k], u = u0[k] + u1[k];
    warp_sum2(g, u);
    if (lane == k) r = RowSums{rows[k], g, u};
  }
  return r;
}

// One NVFP4 chunk: 32 e2m1 codes (16 bytes) in two 16-element blocks with their
// e4m3 scales, against 32 activations given as fp16 pairs (16 words).
// acc += s0 * sum(block 0) + s1 * sum(block 1); the products e2m1 * fp16 are exact
// in fp32 and the block sums accumulate in fp32.
__device__ __forceinline__ void dot32_fp4(float& acc, const uint4 q, uint32_t sc2, const uint32_t* xh) {
  const uint32_t sf = e4m3x2_to_f16x2(sc2);
  const float s0 = __half2float(__ushort_as_half((unsigned short)(sf & 0xffffu)));
  const float s1 = __half2float(__ushort_as_half((unsigned short)(sf >> 16)));
  const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
  float part[2] = {0.0f, 0.0f};
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
    for (int by = 0; by < 4; ++by) {
      const uint32_t wv = e2m1x2_to_f16x2((qw[wi] >> (8 * by)) & 0xffu);
      const uint32_t xv = xh[wi * 4 + by];
      float& pt = part[wi >> 1];
      asm("{\n .reg .b16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %1; mov.b32 {b0, b1}, %2;\n"
          " fma.rn.f32.f16 %0, a0, b0, %0; fma.rn.f32.f16 %0, a1, b1, %0;\n}\n"
          : "+f"(pt)
          : "r"(wv), "r"(xv));
    }
  }
  acc = fmaf(s0, part[0], acc);
  acc = fmaf(s1, part[1], acc);
}

// NVFP4 rows a, b (codes qa, qb; scales sa, sb) against one x row held in the
// lane's registers as fp16 (16 words per 32-element chunk).
__device__ __forceinline__ RowSums dot_one_fp4(const uint4* qa, const uint4* qb, const uint16_t* sa,
                                               const uint16_t* sb, int nch, const uint32_t* xr, int lane) {
  RowSums r{0, 0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < kCplFp4; ++i) {
    const int ch = lane + 32 * i;
    if (ch < nch) {
      dot32_fp4(r.g, qa[ch], sa[ch], xr + 16 * i);
      dot32_fp4(r.u, qb[ch], sb[ch], xr + 16 * i);
    }
  }
  warp_sum2(r.g, r.u);
  if (lane != 0) r.m = -1;
  return r;
}

// NVFP4 rows a, b against the N fp16 x rows of `mask` in shared memory.
template <int N>
__device__ __forceinline__ RowSums dot_rows_fp4(const uint4* qa, const uint4* qb, const uint16_t* sa,
                                                const uint16_t* sb, int nch, const uint4* xs, int H,
                                                uint32_t mask, int lane) {
  int rows[N];
  const uint4* xp[N];
  uint32_t msk = mask;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    rows[k] = __ffs(msk) - 1;
    msk &= msk - 1;
    xp[k] = xs + (size_t)rows[k] * (H / 8);
  }
  float g[N], u[N];
#pragma unroll
  for (int k = 0; k < N; ++k) g[k] = u[k] = 0.0f;
  for (int ch = lane; ch < nch; ch += 32) {
    const uint4 va = qa[ch], vb = qb[ch];
    const uint32_t s_a = sa[ch], s_b = sb[ch];
#pragma unroll
    for (int k = 0; k < N; ++k) {
      uint32_t xh[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = xp[k][ch * 4 + q];
        xh[4 * q] = v.x;
        xh[4 * q + 1] = v.y;
        xh[4 * q + 2] = v.z;
        xh[4 * q + 3] = v.w;
      }
      dot32_fp4(g[k], va, s_a, xh);
      dot32_fp4(u[k], vb, s_b, xh);
    }
  }
  RowSums r{-1, 0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < N; ++k) {
    warp_sum2(g[k], u[k]);
    if (lane == k) r = RowSums{rows[k], g[k], u[k]};
  }
  return r;
}

// One FP8 chunk: 16 e4m3 codes (16 bytes, element k in byte k) against 16
// activations given as fp16 pairs (8 words). Every product e4m3 * fp16 is exact
// in fp32; the sum is fp32. The caller applies the chunk's 128 x 128 block scale.
__device__ __forceinline__ float dot16_fp8(const uint4 q, const uint32_t* xh) {
  const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
  float part = 0.0f;
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const uint32_t wv = e4m3x2_to_f16x2((qw[wi] >> (16 * hb)) & 0xffffu);
      const uint32_t xv = xh[wi * 2 + hb];
      asm("{\n .reg .b16 a0, a1, b0, b1;\n mov.b32 {a0, a1}, %1; mov.b32 {b0, b1}, %2;\n"
          " fma.rn.f32.f16 %0, a0, b0, %0; fma.rn.f32.f16 %0, a1, b1, %0;\n}\n"
          : "+f"(part)
          : "r"(wv), "r"(xv));
    }
  }
  return part;
}

// First fp32 block scale of gate/up row j (j < 2I) of expert e (shared expert
// -1 - e when e < 0): scales are [experts][2I / 128][H / 128].
__device__ __forceinline__ const float* fp8_scale_row13(const Params& p, int e, int j) {
  const float* base = reinterpret_cast<const float*>(e >= 0 ? p.w13_s : p.sh_w13_s);
  const int ex = e >= 0 ? e : -1 - e;
  const int nb = p.H / kFp8Block;
  return base + ((size_t)ex * (2 * p.I / kFp8Block) + j / kFp8Block) * nb;
}

// FP8 rows a, b (codes qa, qb) against one x row held in the lane's registers as
// fp16 (8 words per 16-element chunk); sg, su: the lane's block scales.
__device__ __forceinline__ RowSums dot_one_fp8(const uint4* qa, const uint4* qb, const float* sg, const float* su,
                                               int nch, const uint32_t* xr, int lane) {
  RowSums r{0, 0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < kCplFp8; ++i) {
    const int ch = lane + 32 * i;
    if (ch < nch) {
      r.g = fmaf(sg[i], dot16_fp8(qa[ch], xr + 8 * i), r.g);
      r.u = fmaf(su[i], dot16_fp8(qb[ch], xr + 8 * i), r.u);
    }
  }
  warp_sum2(r.g, r.u);
  if (lane != 0) r.m = -1;
  return r;
}

// FP8 rows a, b against the N fp16 x rows of `mask` in shared memory; the block
// scales are read from the rows' scale vectors (gsr, usr: in the stage, or global).
template <int N>
__device__ __forceinline__ RowSums dot_rows_fp8(const uint4* qa, const uint4* qb, const float* gsr, const float* usr,
                                                int nch, const uint4* xs, int H, uint32_t mask, int lane) {
  int rows[N];
  const uint4* xp[N];
  uint32_t msk = mask;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    rows[k] = __ffs(msk) - 1;
    msk &= msk - 1;
    xp[k] = xs + (size_t)rows[k] * (H / 8);
  }
  float g[N], u[N];
#pragma unroll
  for (int k = 0; k < N; ++k) g[k] = u[k] = 0.0f;
  for (int ch = lane; ch < nch; ch += 32) {
    const uint4 va = qa[ch], vb = qb[ch];
    const float s_a = gsr[ch / 8], s_b = usr[ch / 8];  // global or shared memory
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const uint4 x0 = xp[k][ch * 2], x1 = xp[k][ch * 2 + 1];
      const uint32_t xh[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      g[k] = fmaf(s_a, dot16_fp8(va, xh), g[k]);
      u[k] = fmaf(s_b, dot16_fp8(vb, xh), u[k]);
    }
  }
  RowSums r{-1, 0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < N; ++k) {
    warp_sum2(g[k], u[k]);
    if (lane == k) r = RowSums{rows[k], g[k], u[k]};
  }
  return r;
}

// FP8 block scales of one gate/up item: the gate and up rows' scale vectors, and
// the lane's scales for the register path (loaded before the stage is waited for).
struct Fp8Scales {
  const float* g_row = nullptr;
  const float* u_row = nullptr;
  float gv[kCplFp8], uv[kCplFp8];
};

// The item's gate/up sums: the register path for single-row kernels, else the
// N-row path for the item's row count.
template <int FMT, int MAXM>
__device__ __forceinline__ RowSums item_dot(const uint8_t* st, int iq, int nq, const Params& p,
                                            const uint4* xb, const uint32_t* xh, const uint4* xs, uint32_t mask,
                                            int lane, const Fp8Scales& fs) {
  if (FMT == FMT_BF16) {
    const uint4* wa = reinterpret_cast<const uint4*>(st + (size_t)iq * p.row13);
    const uint4* wb = reinterpret_cast<const uint4*>(st + (size_t)(nq + iq) * p.row13);
    const int nch = p.nchunk_h;
    if constexpr (MAXM == 1) {
      return dot_one_bf16(wa, wb, nch, xb, lane);
    } else {
      switch (__popc(mask)) {
        case 1: return dot_rows_bf16<1>(wa, wb, nch, xs, mask, lane);
        case 2: return dot_rows_bf16<2>(wa, wb, nch, xs, mask, lane);
        case 3: return dot_rows_bf16<3>(wa, wb, nch, xs, mask, lane);
        case 4: return dot_rows_bf16<4>(wa, wb, nch, xs, mask, lane);
        case 5: return dot_rows_bf16<5>(wa, wb, nch, xs, mask, lane);
        case 6: return dot_rows_bf16<6>(wa, wb, nch, xs, mask, lane);
        case 7: return dot_rows_bf16<7>(wa, wb, nch, xs, mask, lane);
        case 8: return dot_rows_bf16<8>(wa, wb, nch, xs, mask, lane);
        default: return RowSums{-1, 0.0f, 0.0f};
      }
    }
  } else if (FMT == FMT_FP8) {
    const uint4* qa = reinterpret_cast<const uint4*>(st + (size_t)iq * p.row13);
    const uint4* qb = reinterpret_cast<const uint4*>(st + (size_t)(nq + iq) * p.row13);
    const int nch = p.nchunk_h;
    if constexpr (MAXM == 1) {
      return dot_one_fp8(qa, qb, fs.gv, fs.uv, nch, xh, lane);
    } else {
      switch (__popc(mask)) {
        case 1: return dot_rows_fp8<1>(qa, qb, fs.g_row, fs.u_row, nch, xs, p.H, mask, lane);
        case 2: return dot_rows_fp8<2>(qa, qb, fs.g_row, fs.u_row, nch, xs, p.H, mask, lane);
        case 3: return dot_rows_fp8<3>(qa, qb, fs.g_row, fs.u_row, nch, xs, p.H, mask, lane);
        case 4: return dot_rows_fp8<4>(qa, qb, fs.g_row, fs.u_row, nch, xs, p.H, mask, lane);
        case 5: return dot_rows_fp8<5>(qa, qb, fs.g_row, fs.u_row, nch, xs, p.H, mask, lane);
        case 6: return dot_rows_fp8<6>(qa, qb, fs.g_row, fs.u_row, nch, xs, p.H, mask, lane);
        case 7: return dot_rows_fp8<7>(qa, qb, fs.g_row, fs.u_row, nch, xs, p.H, mask, lane);
        case 8: return dot_rows_fp8<8>(qa, qb, fs.g_row, fs.u_row, nch, xs, p.H, mask, lane);
        default: return RowSums{-1, 0.0f, 0.0f};
      }
    }
  } else {
    const uint4* qa = reinterpret_cast<const uint4*>(st + (size_t)iq * p.row13);
    const uint4* qb = reinterpret_cast<const uint4*>(st + (size_t)(nq + iq) * p.row13);
    const uint8_t* scb = st + (size_t)2 * nq * p.row13;
    const uint16_t* sa = reinterpret_cast<const uint16_t*>(scb + (size_t)iq * p.sc13);
    const uint16_t* sb = reinterpret_cast<const uint16_t*>(scb + (size_t)(nq + iq) * p.sc13);
    const int nch = p.nchunk_h;
    if constexpr (MAXM == 1) {
      return dot_one_fp4(qa, qb, sa, sb, nch, xh, lane);
    } else {
      switch (__popc(mask)) {
        case 1: return dot_rows_fp4<1>(qa, qb, sa, sb, nch, xs, p.H, mask, lane);
        case 2: return dot_rows_fp4<2>(qa, qb, sa, sb, nch, xs, p.H, mask, lane);
        case 3: return dot_rows_fp4<3>(qa, qb, sa, sb, nch, xs, p.H, mask, lane);
        case 4: return dot_rows_fp4<4>(qa, qb, sa, sb, nch, xs, p.H, mask, lane);
        case 5: return dot_rows_fp4<5>(qa, qb, sa, sb, nch, xs, p.H, mask, lane);
        case 6: return dot_rows_fp4<6>(qa, qb, sa, sb, nch, xs, p.H, mask, lane);
        case 7: return dot_rows_fp4<7>(qa, qb, sa, sb, nch, xs, p.H, mask, lane);
        case 8: return dot_rows_fp4<8>(qa, qb, sa, sb, nch, xs, p.H, mask, lane);
        default: return RowSums{-1, 0.0f, 0.0f};
      }
    }
  }
}

// --------------------------------------------------------------------------
// consumer phases R and U
// --------------------------------------------------------------------------
template <int FMT, int MAXM>
struct XRegs {
  // MAXM == 1: the lane's x chunks, loaded once per phase.
  uint4 b[(MAXM == 1 && FMT == FMT_BF16) ? kCplBf16 : 1];          // bf16 chunks
  uint32_t h[(MAXM == 1 && FMT != FMT_BF16) ? 16 * kCplFp4 : 1];  // fp16 chunks (NVFP4, FP8: 64 words)
};

template <int FMT, int MAXM>
__device__ __forceinline__ void load_xregs(const Ctx& c, XRegs<FMT, MAXM>& xr) {
  if (MAXM != 1) return;
  const Params& p = c.p;
  const uint4* xs = reinterpret_cast<const uint4*>(c.sm + p.off_x);
  const int nch8 = p.H / 8;
  if (FMT == FMT_BF16) {
#pragma unroll
    for (int i = 0; i < kCplBf16; ++i) {
      const int ch = c.lane + 32 * i;
      xr.b[i] = ch < nch8 ? xs[ch] : make_uint4(0, 0, 0, 0);
    }
  } else if (FMT == FMT_FP8) {  // x rows are fp16 by now: 16-element chunks, 8 words each
#pragma unroll
    for (int i = 0; i < kCplFp8; ++i) {
      const int ch = c.lane + 32 * i;
      if (ch < p.H / 16) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint4 v = xs[ch * 2 + q];
          xr.h[8 * i + 4 * q] = v.x;
          xr.h[8 * i + 4 * q + 1] = v.y;
          xr.h[8 * i + 4 * q + 2] = v.z;
          xr.h[8 * i + 4 * q + 3] = v.w;
        }
      }
    }
  } else {  // x rows are fp16 by now
#pragma unroll
    for (int i = 0; i < kCplFp4; ++i) {
      const int ch = c.lane + 32 * i;  // 32-element chunk
      if (ch < p.H / 32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = xs[ch * 4 + q];
          xr.h[16 * i + 4 * q] = v.x;
          xr.h[16 * i + 4 * q + 1] = v.y;
          xr.h[16 * i + 4 * q + 2] = v.z;
          xr.h[16 * i + 4 * q + 3] = v.w;
        }
      }
    }
  }
}

// Power-of-two exponent k that puts a row whose largest |x| has bf16 bits
// `maxbits` into [2^14, 2^15): x * 2^k is then inside fp16's range, and every
// bf16 value of the row down to 2^-29 of the maximum keeps all its bits in fp16
// (smaller ones are below the fp32 rounding of any sum the maximum enters).
__device__ __forceinline__ int xscale_exp(uint32_t maxbits) {
  const int e = (int)(maxbits >> 7);
  if (maxbits == 0u) return 0;
  if (e == 0) return 14 + 133 - (31 - __clz(maxbits & 0x7fu));  // bf16 subnormal: mantissa * 2^-133
  return 14 - (e - 127);
}

// NVFP4 experts multiply e2m1 codes (exact in fp16) with fp16 activations:
// once the bf16 router no longer needs them, the CTA's x rows are converted in
// place, each row scaled by its power of two 2^k (xscale_exp) so that no value
// overflows or loses bits to fp16's smaller exponent range; the gate/up sums are
// scaled back by 2^-k, exactly.
static __device__ __forceinline__ void x_to_f16(const Ctx& c) {
  uint32_t* xw = reinterpret_cast<uint32_t*>(c.sm + c.p.off_x);
  const uint32_t* xmax = reinterpret_cast<const uint32_t*>(c.misc + MISC_XMAX);  // prepare_x(row_max)
  const int hw = c.p.H / 2;  // words per row
  for (int m = 0; m < c.p.M; ++m) {
    // 2^k as two exact factors, each inside fp32's normal range (|k| <= 147)
    const int k = xscale_exp(xmax[m]), k1 = k / 2, k2 = k - k1;
    const float s1 = __int_as_float((k1 + 127) << 23), s2 = __int_as_float((k2 + 127) << 23);
    for (int i = c.tid; i < hw; i += kNC * 32) {
      const uint32_t v = xw[m * hw + i];
      const __half2 h = __floats2half2_rn(bf16lo(v) * s1 * s2, bf16hi(v) * s1 * s2);
      xw[m * hw + i] = *reinterpret_cast<const uint32_t*>(&h);
    }
  }
}

// Router stages: the router logits are on the critical path of every CTA (all
// of them wait for all logits), so the CTA's few router rows are each split
// over several consumer warps along H; the partial sums meet in shared memory.
template <int MAXM>
__device__ __forceinline__ Ring consume_router(const Ctx& c, Ring ring) {
  const Params& p = c.p;
  int lo, hi;
  split_range(p.E / 2, blockIdx.x, p.grid, lo, hi);
  const uint4* xs = reinterpret_cast<const uint4*>(c.sm + p.off_x);
  float* part = reinterpret_cast<float*>(c.sm + p.off_red);  // [kNC][8]
  const uint32_t ep = c.epoch();
  const int nch = p.H / 8;
  ring.fit(p.nslots);
  for (ItemWalk w(lo, hi, p.qr, 0); w.more(); ring.next(p.nslots)) {
    const int nq = w.count();
    const int nrow = 2 * nq;  // <= kNC: the planner keeps qr <= kNC / 2
    const int ws = kNC / nrow;
    const int row = c.warp / ws, seg = c.warp % ws;
    float acc[MAXM];
#pragma unroll
    for (int m = 0; m < MAXM; ++m) acc[m] = 0.0f;
    if (row < nrow && !c.aborted() && c.wait_full(ring)) {
      const uint4* wr = reinterpret_cast<const uint4*>(c.slot_ptr(ring.slot) + (size_t)row * 2 * p.H);
      const int c0 = seg * nch / ws, c1 = (seg + 1) * nch / ws;
      for (int ch = c0 + c.lane; ch < c1; ch += 32) {
        const uint4 wv = wr[ch];
#pragma unroll
        for (int m = 0; m < MAXM; ++m)
          if (m < p.M) dot8_bf16(acc[m], wv, xs[m * nch + ch]);
      }
#pragma unroll
      for (int m = 0; m < MAXM; ++m)
#pragma unroll
        for (int o = 16; o; o >>= 1) acc[m] += __shfl_xor_sync(kFull, acc[m], o);
      if (c.lane == 0)
#pragma unroll
        for (int m = 0; m < MAXM; ++m) part[c.warp * 8 + m] = acc[m];
    }
    bar_sync(kBarConsumers, kNC * 32);  // every partial sum of the stage is in `part`
    if (c.lane == 0) c.release(ring, 1);
    for (int t = c.tid; t < nrow * p.M; t += kNC * 32) {
      const int r = t / p.M, m = t % p.M;
      float v = 0.0f;
      for (int s = 0; s < ws; ++s) v += part[(r * ws + s) * 8 + m];
      if (!(p.test_flags & TEST_SKIP_LOGITS)) {
        const int e = 2 * w.a + r;
#pragma unroll
        for (int rep = 0; rep < kLogitRep; ++rep)
          st_tagged(p.logits + ((size_t)rep * p.maxm + m) * p.E + e, ep, v);
      }
    }
    bar_sync(kBarConsumers, kNC * 32);  // `part` is free again
    w.advance(nq);
  }
  return ring;
}

// The items of one gate/up stage that fall to this warp: dot products against
// the x rows that chose the expert, SwiGLU and the combine weight, h stored in
// pair order (four copies); the slot is handed back for the absent warps too.
template <int FMT, int MAXM>
// hsk / htag (split-K schedule): the h values go to this CTA's shared-memory rows
// (hsk[iq * maxm + m], the stage's first row at hsk) and the row's tag is set once
// they are stored, instead of to the global h rows.
__device__ __forceinline__ void item_stage(const Ctx& c, const Route& rt, const ItemWalk& w, const Ring& ring,
                                           int slot, bool shared, const XRegs<FMT, MAXM>& xr, const uint4* xs,
                                           bool first, float* hsk = nullptr, volatile int* htag = nullptr) {
  const Params& p = c.p;
  const size_t rep_stride = (size_t)p.npair_max * p.I;
  const int nq = w.count();
  const int iq = w.offset(c.warp);
  Fp8Scales fs;
  if (FMT == FMT_FP8 && iq < nq && !p.sc13e) {
    // the item's block scales from global memory, requested before the stage is waited for
    const int e = shared ? -1 - slot : rt.slot_e[slot];
    fs.g_row = fp8_scale_row13(p, e, w.j + iq);
    fs.u_row = fp8_scale_row13(p, e, p.I + w.j + iq);
    if (MAXM == 1) {
#pragma unroll
      for (int i = 0; i < kCplFp8; ++i) {
        const int ch = min(c.lane + 32 * i, p.nchunk_h - 1);
        fs.gv[i] = __ldg(fs.g_row + ch / 8);
        fs.uv[i] = __ldg(fs.u_row + ch / 8);
      }
    }
  }
  if (iq < nq && !c.aborted() && c.wait_full(ring)) {
    if (c.warp == 0 && c.lane == 0 && first) c.stamp(ST_U_DATA);
    const uint8_t* st = c.slot_ptr(ring.slot);
    const int j = w.j + iq;
    if (FMT == FMT_FP8 && p.sc13e) {
      // the expert's scales behind the stage's rows: [2I / 128][H / 128]
      const float* scl = reinterpret_cast<const float*>(st + (size_t)2 * nq * p.row13);
      const int nb = p.H / kFp8Block;
      fs.g_row = scl + (j / kFp8Block) * nb;
      fs.u_row = scl + ((p.I + j) / kFp8Block) * nb;
      if (MAXM == 1) {
#pragma unroll
        for (int i = 0; i < kCplFp8; ++i) {
          const int ch = min(c.lane + 32 * i, p.nchunk_h - 1);
          fs.gv[i] = fs.g_row[ch / 8];
          fs.uv[i] = fs.u_row[ch / 8];
        }
      }
    }
    const uint32_t mask = shared ? (1u << p.M) - 1u : rt.slot_mask[slot];
    const RowSums rs = item_dot<FMT, MAXM>(st, iq, nq, p, xr.b, xr.h, xs, mask, c.lane, fs);
    float gsg = 1.0f, gsu = 1.0f, gs2 = 1.0f;
    int xk = 0;  // NVFP4 / FP8: the row's power-of-two scale of x (x_to_f16)
    if (FMT == FMT_NVFP4) {
      const int e = shared ? -1 - slot : rt.slot_e[slot];
      const float* gs = e >= 0 ? p.w13_gs + 2 * e : p.sh_w13_gs + 2 * (-1 - e);
      gsg = gs[0];
      gsu = gs[1];
      gs2 = e >= 0 ? p.w2_gs[e] : p.sh_w2_gs[-1 - e];  // the down weights' tensor scale, applied once here
    }
    if (rs.m >= 0) {
      if (FMT != FMT_BF16) xk = xscale_exp(reinterpret_cast<const uint32_t*>(c.misc + MISC_XMAX)[rs.m]);
      // 2^-k as two exact factors (each inside fp32's normal range)
      const float q1 = __int_as_float((127 - xk / 2) << 23), q2 = __int_as_float((127 - (xk - xk / 2)) << 23);
      float h = FMT != FMT_BF16 ? silu_f32(rs.g * q1 * q2 * gsg) * (rs.u * q1 * q2 * gsu)
                                : silu_f32(rs.g * gsg) * (rs.u * gsu);
      if (!shared) h *= rt.slot_w[slot * p.maxm + rs.m];
      if (FMT == FMT_NVFP4) h *= gs2;
      if (hsk) {
        hsk[iq * p.maxm + rs.m] = h;
      } else {
      // pair index: a shared slot holds every row (pairs s * M + m); a routed
      // slot's rows follow its pair base in ascending order
      const int pair = shared ? slot * p.M + rs.m : rt.pair_base[slot] + __popc(mask & ((1u << rs.m) - 1u));
      // NVFP4: within a pair the values are interleaved for the down phase's
      // 32-element chunks (element e of chunk c at (e / 4) * 4 * tg + 4 * c + e % 4),
      // so each 16-byte read of a warp is contiguous; bf16 keeps the natural order
      size_t at = (size_t)pair * p.I + j;
      if (FMT == FMT_NVFP4) at = (size_t)pair * p.I + (size_t)((j % 32) >> 2) * (4 * p.tg) + 4 * (j / 32) + (j & 3);
#pragma unroll
      for (int r = 0; r < kHRep; ++r) p.hbuf[r * rep_stride + at] = h;
      }
    }
    __syncwarp();
    if (c.lane == 0) {
      if (htag) {
        __threadfence_block();  // the row's h values (every lane's, ordered by the warp barrier) before its tag
        htag[iq] = 1;
      }
      c.release(ring, iq == 0 ? (uint32_t)(kNC - nq + 1) : 1u);
    }
  }
}

enum ItemKind : int { ITEM_SHARED = 1, ITEM_ROUTED = 2 };

// One phase of gate/up items (shared experts' or routed experts' row pairs):
// each consumer warp takes its items of every stage, computes the dot products
// against the rows of x that chose the expert and publishes tagged h values.
// Returns the ring position after the phase.
// Warps w0 .. w0 + nw - 1 take the items, in stages of q items (0: the planned
// stage size); the other warps walk the same stages without items.
template <int FMT, int MAXM>
__device__ __forceinline__ Ring consume_items(const Ctx& c, const Route& rt, int kind, Ring ring, int w0 = 0,
                                              int nw = kNC, int q = 0) {
  const Params& p = c.p;
  int lo, hi;
  if (kind == ITEM_SHARED) {
    split_range(p.S * p.I, blockIdx.x, p.grid, lo, hi);
  } else {
    lo = c.misc[MISC_ULO];
    hi = c.misc[MISC_UHI];
  }
  const uint4* xs = reinterpret_cast<const uint4*>(c.sm + p.off_x);
  const int slot0 = kind == ITEM_ROUTED ? p.S : 0;
  XRegs<FMT, MAXM> xr;
  load_xregs<FMT, MAXM>(c, xr);
  const int nsl_ring = kind == ITEM_ROUTED ? p.nslots + p.nslots_x : p.nslots;
  ring.fit(nsl_ring);
  ItemWalk w(lo, hi, q > 0 ? q : p.q, p.I);
  w.w0 = w0;
  w.nw = nw;
  for (; w.more(); ring.next(nsl_ring)) {
    item_stage<FMT, MAXM>(c, rt, w, ring, w.u + slot0, kind == ITEM_SHARED, xr, xs, w.a == lo);
    w.advance(w.count());
  }
  return ring;
}

// --------------------------------------------------------------------------
// consumer phase T: top-k per row and the expert union
// --------------------------------------------------------------------------
// Copies n 16-byte units of tagged words (two fp32 values each) from src to dst
// in shared memory: each of the nthr calling threads keeps kStageBatch loads in
// flight and re-polls only the units whose tag is not current yet. False on
// abort / timeout.
static __device__ __forceinline__ bool stage_tagged(const Ctx& c, const unsigned long long* src, float* dst, int n,
                                                 uint32_t site, int nthr) {
  const uint32_t ep = c.epoch();
  uint32_t spins = 0;
  for (int base = c.tid; base < n; base += nthr * kStageBatch) {
    uint32_t pending = 0;
#pragma unroll
    for (int k = 0; k < kStageBatch; ++k)
      if (base + k * nthr < n) pending |= 1u << k;
    while (pending) {
      unsigned long long v0[kStageBatch], v1[kStageBatch];
#pragma unroll
      for (int k = 0; k < kStageBatch; ++k) {
        v0[k] = v1[k] = 0;
        if (pending >> k & 1u) ld_tagged2(src + 2 * (base + k * nthr), v0[k], v1[k]);
      }
#pragma unroll
      for (int k = 0; k < kStageBatch; ++k) {
        if ((pending >> k & 1u) && (uint32_t)(v0[k] >> 32) == ep && (uint32_t)(v1[k] >> 32) == ep) {
          const int u = base + k * nthr;
          dst[2 * u] = __uint_as_float((uint32_t)v0[k]);
          dst[2 * u + 1] = __uint_as_float((uint32_t)v1[k]);
          pending &= ~(1u << k);
        }
      }
      if (!pending) break;
      __nanosleep(64);
      if ((++spins & 15) == 0) {
        if (c.aborted() || c.peer_failed()) return false;
        if (c.expired()) {
          c.fail(site);
          return false;
        }
      }
    }
  }
  return true;
}

// Packed key of expert e with logit v: (order-preserving bits << 32) | ~e, so
// the larger logit wins and equal logits go to the lower expert id. 0 = none.
__device__ __forceinline__ unsigned long long pack_key(float v, int e) {
  return ((unsigned long long)f32_order_key(v) << 32) | (uint32_t)(0xffffffffu - (uint32_t)e);
}
__device__ __forceinline__ int key_expert(unsigned long long k) { return (int)(0xffffffffu - (uint32_t)k); }
__device__ __forceinline__ float key_value(unsigned long long k) { return order_key_f32((uint32_t)(k >> 32)); }

__device__ __forceinline__ unsigned long long shfl_u64(unsigned long long v, int src) {
  const uint32_t lo = __shfl_sync(kFull, (uint32_t)v, src), hi = __shfl_sync(kFull, (uint32_t)(v >> 32), src);
  return ((unsigned long long)hi << 32) | lo;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
  const uint32_t hi = warp_max_u32((uint32_t)(v >> 32));
  const uint32_t lo = warp_max_u32((uint32_t)(v >> 32) == hi ? (uint32_t)v : 0u);
  return ((unsigned long long)hi << 32) | lo;
}
__device__ __forceinline__ float sigmoid_f32(float v) { return 1.0f / (1.0f + expf(-v)); }

// Row m's top-k on warp m from the logits staged in shared memory (lg[e]), with
// every expert's selection key in registers (lane l holds experts l + 32 i,
// PM * 32 >= E). The K-th largest of the 32 lane maxima bounds the K-th largest
// key from below -- those K lane maxima are K distinct experts -- so every
// selected expert's key is at or above it. It is found by K rounds of a
// warp-wide maximum (redux) over the lane maxima, each round retiring the lanes
// that hold the round's value (lanes tied on a value leave together, which can
// only lower the bound); the first round gives the largest key. The few
// candidates at or above the bound go to shared memory at positions given by an
// exclusive count over the lanes (built from ballots of the count's bits), and
// each is ranked against all of them on exact 64-bit keys (ties: the lower
// expert id); the lane that ranks a selected expert also computes its weight
// numerator. With more than kCandMax - 1 candidates (many keys tied in value), K
// rounds of a warp-wide maximum select instead. On this path one warp's
// dependent chain is the routing latency every CTA waits for, so it uses
// reductions and ballots rather than shuffles, and shared memory where a value
// must reach every lane. The expert row masks (rt.emask) are set for M > 1 only.
template <int PM>
__device__ __forceinline__ void topk_row(const Ctx& c, const Route& rt, int m, bool write_topk) {
  const Params& p = c.p;
  const int E = p.E, K = p.K, lane = c.lane;
  const float* lg = reinterpret_cast<const float*>(c.sm + p.off_lg) + (size_t)m * E;
  const float* bias = reinterpret_cast<const float*>(c.sm + p.off_bias);
  float* wx = reinterpret_cast<float*>(c.sm + p.off_lmax) + m * 32;  // numerators of the weights, by rank
  unsigned long long* cand = reinterpret_cast<unsigned long long*>(c.sm + p.off_cand) + (size_t)m * kCandMax;
  uint32_t key[PM];
  if (p.score) {  // bias-corrected sigmoid rule: select on sigmoid(l) + b
#pragma unroll
    for (int i = 0; i < PM; ++i) {
      const int e = lane + 32 * i;
      key[i] = e < E ? f32_order_key(sigmoid_f32(lg[e]) + bias[e]) : 0u;
    }
  } else {
#pragma unroll
    for (int i = 0; i < PM; ++i) {
      const int e = lane + 32 * i;
      key[i] = e < E ? f32_order_key(lg[e]) : 0u;
    }
  }
  uint32_t t[PM];
#pragma unroll
  for (int i = 0; i < PM; ++i) t[i] = key[i];
#pragma unroll
  for (int h = PM / 2; h >= 1; h >>= 1)
#pragma unroll
    for (int i = 0; i < h; ++i) t[i] = max(t[i], t[i + h]);
  // the bound: K rounds over the lane maxima
  uint32_t lk = t[0];
  const uint32_t Tmax = warp_max_u32(lk);
  uint32_t T = Tmax;
  lk = lk == T ? 0u : lk;
  for (int r = 1; r < K; ++r) {
    T = warp_max_u32(lk);
    lk = lk == T ? 0u : lk;
  }
  uint32_t fm = 0;
#pragma unroll
  for (int i = 0; i < PM; ++i) fm |= (uint32_t)(key[i] >= T && key[i] != 0u) << i;
  // exclusive count of candidates over the lanes, and the total, bit by bit
  const int cnt = __popc(fm);
  const uint32_t lt = (1u << lane) - 1u;
  int o = 0, C = 0;
#pragma unroll
  for (int bit = 0; bit < (PM > 16 ? 6 : 5); ++bit) {
    const uint32_t bb = __ballot_sync(kFull, (cnt >> bit) & 1);
    o += __popc(bb & lt) << bit;
    C += __popc(bb) << bit;
  }
  int* sel_e = rt.sel_e + m * K;
  float* sel_w = rt.sel_w + m * K;
  // weight numerator of a selected key: exp(l - l_max) (softmax rule; l_max is
  // the largest key's logit) or sigmoid(l) (bias rule)
  const float lmax = order_key_f32(Tmax);
  auto numer = [&](unsigned long long v) {
    return p.score ? sigmoid_f32(lg[key_expert(v)]) : expf(key_value(v) - lmax);
  };
  if (C < kCandMax) {
#pragma unroll
    for (int i = 0; i < PM; ++i)
      if (fm >> i & 1u) cand[o++] = ((unsigned long long)key[i] << 32) | (0xffffffffu - (uint32_t)(lane + 32 * i));
    if (lane == 0) cand[C] = 0ull;  // pads the pairwise scan below (no key is 0)
    __syncwarp();
    const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(cand);
    for (int ci = lane; ci < C; ci += 32) {
      const unsigned long long v = cand[ci];
      int r = 0;
#pragma unroll 4
      for (int j = 0; j < (C + 1) / 2; ++j) {
        const ulonglong2 q = c2[j];
        r += (q.x > v) + (q.y > v);
      }
      if (r < K) {
        sel_e[r] = key_expert(v);
        wx[r] = numer(v);
      }
    }
  } else {
    unsigned long long last = ~0ull;
    for (int j = 0; j < K; ++j) {
      unsigned long long b = 0;
#pragma unroll
      for (int i = 0; i < PM; ++i) {
        const unsigned long long k =
            key[i] ? ((unsigned long long)key[i] << 32) | (0xffffffffu - (uint32_t)(lane + 32 * i)) : 0ull;
        if (k < last && k > b) b = k;
      }
      last = warp_max_u64(b);
      if (lane == 0) {
        sel_e[j] = key_expert(last);
        wx[j] = numer(last);
      }
    }
  }
  __syncwarp();
  // weights in selection order: every lane sums the K numerators in order
  float sum = 0.0f;
  for (int j = 0; j < K; ++j) sum += wx[j];
  if (lane < K) {
    const int ej = sel_e[lane];
    const float w = wx[lane] / sum;
    if (p.M > 1) atomicOr(&rt.emask[ej], 1u << m);
    if (write_topk && blockIdx.x == 0) {
      if (p.topk_idx) p.topk_idx[m * K + lane] = ej;
      if (p.topk_w) p.topk_w[m * K + lane] = w;
    }
    sel_w[lane] = w;
  }
}

// The union of the experts chosen by M > 1 rows, one thread per (row, selected
// expert) pair (nthr threads meeting at named barrier `bar`; M * K <= 128 pairs).
// Each pair thread marks whether its row is the lowest one that chose its expert;
// then it counts, over all pairs, the pairs and the distinct experts with a
// smaller id: its slot is S + (distinct experts below), its (slot, row) pair
// index follows the slot's pair base in ascending row order. The thread of each
// expert's lowest row writes the slot's tables and checks whether one of this
// CTA's gate/up cost boundaries falls in its slot's cost interval
// [cum(u), cum(u + 1)), cum(u) = I * (item_base * u + pairs before slot u).
__device__ __forceinline__ void union_rows(const Ctx& c, const Route& rt, int nthr, int bar) {
  const Params& p = c.p;
  const int M = p.M, K = p.K, S = p.S, np = M * K;
  int* psr = reinterpret_cast<int*>(c.sm + p.off_pair_sr);
  int* fl = reinterpret_cast<int*>(c.sm + p.off_cand);  // [np]: expert << 1 | lowest row (the top-k is done with it)
  for (int t = c.tid; t < np; t += nthr) {
    const int e = rt.sel_e[t], m = t / K;
    fl[t] = (e << 1) | (int)(m == __ffs(rt.emask[e]) - 1);
  }
  bar_sync(bar, nthr);
  const uint32_t I = (uint32_t)p.I, base = (uint32_t)p.item_base;
  for (int t = c.tid; t < np; t += nthr) {
    const int e = rt.sel_e[t], m = t / K;
    const uint32_t msk = rt.emask[e];
    int pb = 0, sb = 0, tot = 0;  // pairs and experts below e, experts in all
    const int4* f4 = reinterpret_cast<const int4*>(fl);
    for (int j = 0; j < np / 4; ++j) {
      const int4 q = f4[j];
      const int v[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int below = (v[k] >> 1) < e;
        pb += below;
        sb += below & v[k];
        tot += v[k] & 1;
      }
    }
    for (int j = np & ~3; j < np; ++j) {
      const int v = fl[j], below = (v >> 1) < e;
      pb += below;
      sb += below & v;
      tot += v & 1;
    }
    const int sl = S + sb;
    rt.slot_w[sl * p.maxm + m] = rt.sel_w[t] * p.routed_scale;
    psr[S * M + pb + __popc(msk & ((1u << m) - 1u))] = (sl << 4) | m;
    if (m == __ffs(msk) - 1) {
      rt.slot_of[e] = sl;
      rt.slot_e[sl] = e;
      rt.slot_mask[sl] = msk;
      rt.pair_base[sl] = S * M + pb;
      const uint32_t tcost = I * (base * (uint32_t)tot + (uint32_t)np);  // < 2^24
      const uint32_t t0 = tcost * blockIdx.x / (uint32_t)p.grid, t1 = tcost * (blockIdx.x + 1) / (uint32_t)p.grid;
      const uint32_t wu = base + (uint32_t)__popc(msk);
      const uint32_t cu = I * (base * (uint32_t)sb + (uint32_t)pb), cn = cu + I * wu;
      // each boundary: the first item at or after its cost, in the slot whose interval holds it
      if (cu <= t0 && t0 < cn) c.misc[MISC_ULO] = sb * p.I + (int)((t0 - cu + wu - 1) / wu);
      if (cu <= t1 && t1 < cn) c.misc[MISC_UHI] = sb * p.I + (int)((t1 - cu + wu - 1) / wu);
      if (sb == 0) {  // once: the end of the sequence
        rt.pair_base[S + tot] = S * M + np;
        c.misc[MISC_NROUTED] = tot;
        if (tcost <= t0) c.misc[MISC_ULO] = tot * p.I;
        if (tcost <= t1) c.misc[MISC_UHI] = tot * p.I;
      }
    }
  }
  for (int t = c.tid; t < S; t += nthr) {
    rt.slot_e[t] = -1 - t;
    rt.slot_mask[t] = (1u << M) - 1u;
    rt.pair_base[t] = t * M;
    for (int m = 0; m < p.maxm; ++m) rt.slot_w[t * p.maxm + m] = 1.0f;
    for (int m = 0; m < M; ++m) psr[t * M + m] = (t << 4) | m;
  }
}

// The union for a single token row on warp 0: the K selected experts in
// ascending id become slots S.., one pair each; the same tables as union_rows
// builds. Each lane counts the selected ids below its own from shared memory
// (broadcast loads, no shuffles). The gate/up split bounds of a single row do
// not depend on the routing and were set before it (one_row_split).
__device__ __forceinline__ void union_one_row(const Ctx& c, const Route& rt) {
  const Params& p = c.p;
  const int K = p.K, S = p.S, lane = c.lane;
  int* psr = reinterpret_cast<int*>(c.sm + p.off_pair_sr);
  const int e = lane < K ? rt.sel_e[lane] : 0x7fffffff;
  const int4* s4 = reinterpret_cast<const int4*>(rt.sel_e);  // K <= 16, 16-byte aligned
  int rank = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (4 * j < K) {
      const int4 q = s4[j];
      rank += (q.x < e) + (4 * j + 1 < K && q.y < e) + (4 * j + 2 < K && q.z < e) + (4 * j + 3 < K && q.w < e);
    }
  }
  if (lane < K) {
    const float w = rt.sel_w[lane];
    const int sl = S + rank;
    rt.slot_of[e] = sl;
    rt.slot_e[sl] = e;
    rt.slot_mask[sl] = 1u;
    rt.slot_w[sl * p.maxm] = w * p.routed_scale;
    rt.pair_base[sl] = sl;  // shared slots hold one pair each, so slot and pair index agree
    psr[sl] = sl << 4;
  }
  for (int t = lane; t < S; t += 32) {
    rt.slot_e[t] = -1 - t;
    rt.slot_mask[t] = 1u;
    for (int m = 0; m < p.maxm; ++m) rt.slot_w[t * p.maxm + m] = 1.0f;
    rt.pair_base[t] = t;
    psr[t] = t << 4;
  }
  if (lane == 0) {
    rt.pair_base[S + K] = S + K;
    c.misc[MISC_NROUTED] = K;
  }
}

// A single row's gate/up cost split: every routed item has one row, so it is the
// plain split of K * I items over the CTAs, known before the routing.
__device__ __forceinline__ void one_row_split(const Ctx& c) {
  int lo, hi;
  split_range(c.p.K * c.p.I, blockIdx.x, c.p.grid, lo, hi);
  c.misc[MISC_ULO] = lo;
  c.misc[MISC_UHI] = hi;
}

// The experts the next run of this handle prefetches (speculative expert
// prefetch, off unless pf_n > 0): the routed experts of this run used by the
// most token rows, ties to the lower expert id; with one row, the selected
// experts in selection order (descending weight). Written by warp 0 of CTA 0
// after its work, from the routing tables still in shared memory, into the list
// of the next run's parity.
__device__ __forceinline__ void write_prediction(const Ctx& c, const Route& rt) {
  const Params& p = c.p;
  if (p.pf_n <= 0 || p.hist == nullptr || blockIdx.x != 0 || c.warp != 0) return;
  int* out = p.hist + (size_t)((c.epoch() + 1u) & 1u) * kPfMax;
  const int P = min(p.pf_n, kPfMax);
  if (p.M == 1) {
    if (c.lane < kPfMax) out[c.lane] = c.lane < P && c.lane < p.K ? rt.sel_e[c.lane] : -1;
    return;
  }
  const int nr = c.misc[MISC_NROUTED];
  uint32_t key[4];  // routed slots lane + 32 i: (rows << 16) | (0xffff - slot); 0 = none
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int u = c.lane + 32 * i;
    key[i] = u < nr ? ((uint32_t)__popc(rt.slot_mask[p.S + u]) << 16) | (0xffffu - (uint32_t)u) : 0u;
  }
  for (int j = 0; j < kPfMax; ++j) {
    uint32_t best = 0;
    if (j < P) {
#pragma unroll
      for (int i = 0; i < 4; ++i) best = max(best, key[i]);
      best = warp_max_u32(best);
#pragma unroll
      for (int i = 0; i < 4; ++i) key[i] = key[i] == best ? 0u : key[i];
    }
    if (c.lane == 0) out[j] = best ? rt.slot_e[p.S + (int)(0xffffu - (best & 0xffffu))] : -1;
  }
}

// nthr threads (the first nthr / 32 consumer warps, at least p.M) route; they
// meet at named barrier `bar`. MAXM: the kernel's row bound (MAXM == 1 exactly
// when the run has one row).
template <int MAXM>
static __device__ __forceinline__ void route_rows(const Ctx& c, const Route& rt, bool write_topk,
                                                  int nthr = kNC * 32, int bar = kBarConsumers) {
  const Params& p = c.p;
  // the selection bias (bias-corrected sigmoid rule) into shared memory while
  // the logits are still on their way
  if (p.score) {
    float* bs = reinterpret_cast<float*>(c.sm + p.off_bias);
    for (int e = c.tid; e < p.E; e += nthr) bs[e] = __ldg(p.router_bias + e);
  }
  if (MAXM == 1 && c.tid == 0) one_row_split(c);
  // this CTA's replica of the logits into shared memory (coalesced): every word
  // carries its run tag, so each thread polls its words until the tags are this
  // run's, with no count or flag to wait for first
  float* lg = reinterpret_cast<float*>(c.sm + p.off_lg);
  const unsigned long long* src = p.logits + (size_t)(blockIdx.x % kLogitRep) * p.maxm * p.E;
  bool ok = !c.aborted() && stage_tagged(c, src, lg, p.M * p.E / 2, SITE_LOGITS, nthr);
  if (!ok)  // keep going on well-defined data: outputs are void after a timeout
    for (int i = c.tid; i < p.M * p.E; i += nthr) lg[i] = 0.0f;
  bar_sync(bar, nthr);
  if (c.tid == 0) c.stamp(ST_LOGITS);
  if (c.warp < p.M) {
    if (p.E <= 16 * 32)
      topk_row<16>(c, rt, c.warp, write_topk);
    else
      topk_row<32>(c, rt, c.warp, write_topk);
  }
  bar_sync(bar, nthr);
  if (c.tid == 0) c.stamp(ST_TOPK);
  if constexpr (MAXM == 1) {
    if (c.warp == 0) union_one_row(c, rt);
  } else {
    union_rows(c, rt, nthr, bar);
  }
  bar_sync(bar, nthr);
}

// --------------------------------------------------------------------------
// consumer phase D
// --------------------------------------------------------------------------
__device__ __forceinline__ void cta_rows(const Params& p, int& r_lo, int& r_hi) {
  split_range(p.H, blockIdx.x, p.grid, r_lo, r_hi);
}

// Wait until every CTA has its copy of x (only needed when the output
// overwrites x in the single-kernel schedule).
static __device__ __forceinline__ bool wait_xflags(const Ctx& c) {
  const Params& p = c.p;
  const uint32_t ep = c.epoch();
  uint64_t spins = 0;
  for (int i = c.tid; i < p.grid; i += kNC * 32) {
    for (;;) {
      const unsigned long long v = ld_relaxed_u64(p.xflags + i);
      if ((uint32_t)(v >> 32) == ep) break;
      if (c.aborted() || ((++spins & 63) == 0 && c.peer_failed())) return false;
      if (c.expired()) {
        c.fail(SITE_XFLAGS);
        return false;
      }
    }
  }
  return true;
}

// Per-slot h readiness (every pair fits the h area): this CTA adds the number of
// its gate/up items of each slot to that slot's count; a slot's h is complete
// when its count reaches I. Thread 0, after the CTA's h stores and a fence.
__device__ __forceinline__ void count_slots(const Ctx& c) {
  const Params& p = c.p;
  auto add = [&](int slot0, int lo, int hi) {
    for (int u = lo / p.I; lo < hi; ++u) {
      const int end = min(hi, (u + 1) * p.I);
      asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p.ctrl + CTRL_SLOTCNT + slot0 + u),
                   "r"((uint32_t)(end - lo))
                   : "memory");
      lo = end;
    }
  };
  int slo, shi;
  split_range(p.S * p.I, blockIdx.x, p.grid, slo, shi);
  add(0, slo, shi);
  add(p.S, c.misc[MISC_ULO], c.misc[MISC_UHI]);
}

// Down-phase batches: slots [sl0, sl1) whose (expert, row) pairs fit one h
// buffer of `cap` pairs. With S >= 0 the first S (shared) slots form batches of
// their own (their h is complete long before the routed experts').
__device__ __forceinline__ int batch_end(const Route& rt, int sl0, int nsl, int cap, int S) {
  int sl1 = sl0 + 1;
  while (sl1 < nsl && sl1 != S && rt.pair_base[sl1 + 1] - rt.pair_base[sl0] <= cap) ++sl1;
  return sl1;
}

// The h values of the pairs of slots [sl0, sl1) -- contiguous in pair order --
// from this CTA's copy of the h buffer into shared h buffer b: one bulk copy
// counted on the buffer's mbarrier. Thread 0 only.
__device__ __forceinline__ void issue_h(const Ctx& c, const Route& rt, int sl0, int sl1, int b, int cap) {
  const Params& p = c.p;
  const int p0 = rt.pair_base[sl0];
  const uint32_t bytes = (uint32_t)(rt.pair_base[sl1] - p0) * (uint32_t)p.I * 4u;
  const float* src = p.hbuf + ((size_t)(blockIdx.x % kHRep) * p.npair_max + p0) * p.I;
  float* dst = reinterpret_cast<float*>(c.sm + p.off_hs) + (size_t)b * cap * p.I;
  const uint32_t bar = smem_u32(c.sm + p.off_hbar) + 8u * b;
  mbar_arrive_expect_tx(bar, bytes);
  bulk_g2s_plain(smem_u32(dst), src, bytes, bar);
}

// FP8 down-projection block scales of expert e (shared expert -1 - e when e < 0):
// [H / 128][I / 128] per expert.
__device__ __forceinline__ const float* fp8_scale_down(const Params& p, int e) {
  const float* base = reinterpret_cast<const float*>(e >= 0 ? p.w2_s : p.sh_w2_s);
  return base + (size_t)(e >= 0 ? e : -1 - e) * (p.H / kFp8Block) * (p.I / kFp8Block);
}

// FP8 down scales of expert e for the down stage in ring slot `ring`: staged in the
// slot at d_soff, or the expert's scales in global memory (d: the down-phase slot
// map of the phase-ordered kernel).
__device__ __forceinline__ const float* fp8_down_scales(const Ctx& c, const Ring& ring, bool d, int e) {
  if (!c.p.sc2e) return fp8_scale_down(c.p, e);
  return reinterpret_cast<const float*>(c.slot_ptr(ring.slot, d) + c.p.d_soff);
}

// One down stage: this thread's rows of the CTA's output block (group g, 16-byte
// code chunk ch) against the h rows of the slot's pairs (hs, in pair order),
// accumulated in fp32 over the slots.
// FP8: s2 = the expert's block scales [H / 128][I / 128] (in the stage, or in
// global memory), row0 = the global row of the stage's first row.
template <int FMT, int MAXM>
__device__ __forceinline__ void down_stage(const Params& p, const uint8_t* st, const float* hs, uint32_t mask,
                                           float (&acc)[rows_per_group(FMT)][MAXM], int g, int ch, int nr,
                                           const float* s2 = nullptr, int row0 = 0) {
  constexpr int RPG = rows_per_group(FMT);
  const int drs = p.d_rows_stage;
  int hp = 0;
  float sv[FMT == FMT_FP8 ? RPG : 1];
  if (FMT == FMT_FP8) {  // each row's scale of this thread's 8-code chunk
#pragma unroll
    for (int ri = 0; ri < RPG; ++ri) {
      const int r = min(g + ri * p.ng, nr - 1);
      sv[ri] = s2[(size_t)((row0 + r) / kFp8Block) * (p.I / kFp8Block) + (8 * ch) / kFp8Block];
    }
  }
  if constexpr (FMT == FMT_BF16 && MAXM > 1 && MAXM <= 6) {
    // each weight widened once and used for every row that chose the expert
    // (the registers allow it up to six rows)
    float wf[RPG][8];
#pragma unroll
    for (int ri = 0; ri < RPG; ++ri) {
      const int r = min(g + ri * p.ng, nr - 1);
      const uint4 v = reinterpret_cast<const uint4*>(st + (size_t)r * p.row2)[ch];
      const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        wf[ri][2 * q] = bf16lo(vw[q]);
        wf[ri][2 * q + 1] = bf16hi(vw[q]);
      }
    }
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
      if (!(mask >> m & 1u)) continue;
      const float* hrow = hs + (size_t)hp * p.I;
      ++hp;
      const float4 a = *reinterpret_cast<const float4*>(hrow + 8 * ch);
      const float4 b = *reinterpret_cast<const float4*>(hrow + 8 * ch + 4);
      const float hv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int ri = 0; ri < RPG; ++ri)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[ri][m] = fmaf(wf[ri][k], hv[k], acc[ri][m]);
    }
  } else {
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
      if (!(mask >> m & 1u)) continue;
      const float* hrow = hs + (size_t)hp * p.I;
      ++hp;
      if (FMT == FMT_BF16) {
        const float4 a = *reinterpret_cast<const float4*>(hrow + 8 * ch);
        const float4 b = *reinterpret_cast<const float4*>(hrow + 8 * ch + 4);
        const float hv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        // every row of the group, branch-free: rows past the block repeat
        // the last one (their sums are never written), so all loads issue
        // before the arithmetic
        uint4 wv[RPG];
#pragma unroll
        for (int ri = 0; ri < RPG; ++ri) {
          const int r = min(g + ri * p.ng, nr - 1);
          wv[ri] = reinterpret_cast<const uint4*>(st + (size_t)r * p.row2)[ch];
        }
#pragma unroll
        for (int ri = 0; ri < RPG; ++ri) dot8_bf16_f32(acc[ri][m], wv[ri], hv);
      } else if (FMT == FMT_FP8) {
        // 8 e4m3 codes per thread and row against 8 fp32 h values, summed in
        // fp32 (one rounding per fused multiply-add), then the row's block scale
        const float4 a = *reinterpret_cast<const float4*>(hrow + 8 * ch);
        const float4 b = *reinterpret_cast<const float4*>(hrow + 8 * ch + 4);
        const float hv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint2 wv[RPG];
#pragma unroll
        for (int ri = 0; ri < RPG; ++ri) {
          const int r = min(g + ri * p.ng, nr - 1);
          wv[ri] = reinterpret_cast<const uint2*>(st + (size_t)r * p.row2)[ch];
        }
#pragma unroll
        for (int ri = 0; ri < RPG; ++ri) {
          const uint32_t qw[2] = {wv[ri].x, wv[ri].y};
          float part = 0.0f;
#pragma unroll
          for (int wi = 0; wi < 2; ++wi) {
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              const uint32_t f = e4m3x2_to_f16x2((qw[wi] >> (16 * hb)) & 0xffffu);
              const __half2 w2 = *reinterpret_cast<const __half2*>(&f);
              const int e0 = wi * 4 + hb * 2;
              part = fmaf(__low2float(w2), hv[e0], part);
              part = fmaf(__high2float(w2), hv[e0 + 1], part);
            }
          }
          acc[ri][m] = fmaf(sv[ri], part, acc[ri][m]);
        }
      } else {
        // one 16-element block (one e4m3 scale) at a time: 16 h values in registers
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          float hv[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 f = *reinterpret_cast<const float4*>(hrow + 4 * ch + (blk * 4 + q) * 4 * p.tg);
            hv[4 * q] = f.x;
            hv[4 * q + 1] = f.y;
            hv[4 * q + 2] = f.z;
            hv[4 * q + 3] = f.w;
          }
#pragma unroll
          for (int ri = 0; ri < RPG; ++ri) {
            const int r = g + ri * p.ng;
            if (r < nr) {
              const uint2 qv = reinterpret_cast<const uint2*>(st + (size_t)r * p.row2 + 16 * ch)[blk];
              const uint32_t sb = st[(size_t)drs * p.row2 + (size_t)r * p.sc2 + 2 * ch + blk];
              const float sv = __half2float(__ushort_as_half((unsigned short)(e4m3x2_to_f16x2(sb) & 0xffffu)));
              const uint32_t qw[2] = {qv.x, qv.y};
              float part = 0.0f;
#pragma unroll
              for (int wi = 0; wi < 2; ++wi) {
#pragma unroll
                for (int by = 0; by < 4; ++by) {
                  const uint32_t wv = e2m1x2_to_f16x2((qw[wi] >> (8 * by)) & 0xffu);
                  const int e0 = wi * 8 + by * 2;
                  const __half2 wh = *reinterpret_cast<const __half2*>(&wv);
                  part = fmaf(__low2float(wh), hv[e0], part);
                  part = fmaf(__high2float(wh), hv[e0 + 1], part);
                }
              }
              acc[ri][m] = fmaf(sv, part, acc[ri][m]);
            }
          }
        }
      }
    }
  }
}

// Sums of each output row over the group's threads, plus the residual, rounded
// once to bf16 and stored (rows rb_lo + r, r < nr).
template <int FMT, int MAXM>
__device__ __forceinline__ void write_rows(const Ctx& c, float (&acc)[rows_per_group(FMT)][MAXM], int g, int ch,
                                           bool active, int nr, int rb_lo) {
  const Params& p = c.p;
  constexpr int RPG = rows_per_group(FMT);
  float* red = reinterpret_cast<float*>(c.sm + p.off_red);
  const bool write = !c.aborted();
  if (p.tg <= 32) {
#pragma unroll
    for (int ri = 0; ri < RPG; ++ri)
#pragma unroll
      for (int m = 0; m < MAXM; ++m)
        for (int o = p.tg >> 1; o; o >>= 1) acc[ri][m] += __shfl_xor_sync(kFull, acc[ri][m], o);
    if (write && active && ch == 0) {
#pragma unroll
      for (int ri = 0; ri < RPG; ++ri) {
        const int r = g + ri * p.ng;
        if (r < nr) {
          const int row = rb_lo + r;
#pragma unroll
          for (int m = 0; m < MAXM; ++m) {
            if (m < p.M) {
              const float rv = __uint_as_float((uint32_t)p.resid[(size_t)m * p.H + row] << 16);
              p.out[(size_t)m * p.H + row] = f32_to_bf16_bits(rv + acc[ri][m]);
            }
          }
        }
      }
    }
  } else {
#pragma unroll
    for (int ri = 0; ri < RPG; ++ri)
#pragma unroll
      for (int m = 0; m < MAXM; ++m) {
        float v = acc[ri][m];
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
        if (c.lane == 0) red[(c.warp * RPG + ri) * MAXM + m] = v;
      }
    bar_sync(kBarConsumers, kNC * 32);
    const int wpg = p.tg / 32;
    if (write && active && ch < 32) {  // first warp of each group writes
      for (int q = c.lane; q < RPG * MAXM; q += 32) {
        const int ri = q / MAXM, m = q % MAXM;
        const int r = g + ri * p.ng;
        if (r < nr && m < p.M) {
          float y = 0.0f;
          for (int w = 0; w < wpg; ++w) y += red[((g * wpg + w) * RPG + ri) * MAXM + m];
          const int row = rb_lo + r;
          const float rv = __uint_as_float((uint32_t)p.resid[(size_t)m * p.H + row] << 16);
          p.out[(size_t)m * p.H + row] = f32_to_bf16_bits(rv + y);
        }
      }
    }
    bar_sync(kBarConsumers, kNC * 32);
  }
}

// wait_u: the gate/up results come from this same kernel (single-kernel schedule)
// nd: down-phase slots in the x area (0 or 1)
template <int FMT, int MAXM>
__device__ void consume_down(const Ctx& c, const Route& rt, bool check_xflags, bool wait_u, Ring ring, int nd) {
  const Params& p = c.p;
  int r_lo, r_hi;
  cta_rows(p, r_lo, r_hi);
  const int drs = p.d_rows_stage;
  const int nrb = (r_hi - r_lo + drs - 1) / drs;
  const int nsl = p.S + c.misc[MISC_NROUTED];
  const int ctid = c.tid;
  const int g = ctid / p.tg;   // thread group
  const int ch = ctid % p.tg;  // 16-byte code chunk of a down row
  const bool active = g < p.ng;
  const float* hs0 = reinterpret_cast<const float*>(c.sm + p.off_hs);
  const uint32_t hbar0 = smem_u32(c.sm + p.off_hbar);
  const int nbuf = p.hs_nbuf, cap = p.hs_pairs / nbuf;
  constexpr int RPG = rows_per_group(FMT);  // rows per thread group and stage
  // Thread 0 keeps up to nbuf batches of h in flight: batch uses run over
  // (row block, batch) in order; use u goes to buffer u % nbuf and may be issued
  // once use u - nbuf is done. With two buffers (the pairs do not all fit at
  // once) and wait_u, a batch of shared slots waits only for every CTA's shared
  // h (SCOUNT): the shared experts' down stages run while the last gate/up items
  // finish elsewhere. Every other batch waits for all h (UCOUNT).
  const int split = (wait_u && nbuf == 2) ? p.S : -1;
  int a_rb = 0, a_sl = 0, issued = 0, landed = 0;
  bool s_ok = !wait_u, u_ok = !wait_u;
  auto issue_ready = [&](int limit, bool may_wait) {  // thread 0
    while (issued < limit && a_rb < nrb && !c.aborted()) {
      const bool routed = a_sl >= split;
      bool& ok = routed ? u_ok : s_ok;
      if (!ok) {
        if (!may_wait) return;
        if (!wait_count(c, routed ? CTRL_UCOUNT : CTRL_SCOUNT, SITE_FLAGS)) {
          c.abort_local();
          return;
        }
        if (routed) c.stamp(ST_U_FLAGS);
        __threadfence();             // acquire every CTA's h stores ...
        fence_proxy_async_global();  // ... for the bulk copies that read them
        ok = true;
      }
      const int sl1 = batch_end(rt, a_sl, nsl, cap, split);
      issue_h(c, rt, a_sl, sl1, issued % nbuf, cap);
      ++issued;
      a_sl = sl1;
      if (a_sl >= nsl) {
        a_sl = 0;
        ++a_rb;
      }
    }
  };
  // per-slot mode: one producer lane fetches each slot's h as soon as it is
  // complete (fetch_h_per_slot); all pairs stay in the h area for every row block
  const bool per_slot = wait_u && p.hs_perslot;
  if (nrb > 0 && !per_slot) {
    fence_proxy_async_shared();  // generic accesses to the h area (routing scratch) before the copies into it
    bar_sync(kBarConsumers, kNC * 32);
    if (c.tid == 0) issue_ready(1, true);           // the first batch, waiting as needed
    if (c.tid == 0) issue_ready(nbuf, split <= 0);  // more without waiting for the routed h
  }
  int used = 0;
  ring.fit(p.nslots + nd);
  for (int rb = 0; rb < nrb; ++rb) {
    const int rb_lo = r_lo + rb * drs;
    const int nr = min(drs, r_hi - rb_lo);
    float acc[RPG][MAXM];
#pragma unroll
    for (int ri = 0; ri < RPG; ++ri)
#pragma unroll
      for (int m = 0; m < MAXM; ++m) acc[ri][m] = 0.0f;
    for (int sl0 = 0; sl0 < nsl;) {
      const int sl1 = batch_end(rt, sl0, nsl, cap, split);
      const int b = used % nbuf;
      bool have = true;
      if (!per_slot) {
        if (c.tid == 0) issue_ready(used + nbuf, true);  // this batch if it was held back, and the next
        const uint64_t th = p.stamps ? global_ns() : 0;
        have = !c.aborted() && c.wait_bar(hbar0 + 8u * b, (uint32_t)(used / nbuf) & 1u, SITE_HIDDEN);
        if (p.stamps && c.tid == 0) c.count(ST_D_HWAIT_NS, global_ns() - th);
        if (have && c.tid == 0) landed = used + 1;
      }
      const float* hs = hs0 + (size_t)b * cap * p.I;
      if (rb == 0 && sl0 == 0 && c.tid == 0) c.stamp(ST_D_FIRST);
      for (int sl = sl0; sl < sl1; ++sl, ring.next(p.nslots + nd)) {
        const uint32_t mask = rt.slot_mask[sl];
        if (per_slot && rb == 0) {  // this slot's h (once: it stays for later row blocks)
          const uint64_t th = p.stamps ? global_ns() : 0;
          have = !c.aborted() && c.wait_bar(c.full0 + 8u * (kHSlotBar + sl), 0, SITE_HIDDEN);
          if (p.stamps && c.tid == 0) c.count(ST_D_HWAIT_NS, global_ns() - th);
        }
        const uint64_t tw = p.stamps ? global_ns() : 0;
        const bool got = !c.aborted() && c.wait_full(ring);
        const uint64_t tm = p.stamps ? global_ns() : 0;
        if (p.stamps && c.tid == 0) c.count(ST_D_WAIT_NS, tm - tw);
        if (got && have && active)
          down_stage<FMT, MAXM>(p, c.slot_ptr(ring.slot, true), hs + (size_t)(rt.pair_base[sl] - rt.pair_base[sl0]) * p.I,
                                mask, acc, g, ch, nr, fp8_down_scales(c, ring, true, sl < p.S ? -1 - sl : rt.slot_e[sl]),
                                rb_lo);
        __syncwarp();
        if (p.stamps && c.tid == 0) c.count(ST_D_MATH_NS, global_ns() - tm);
        if (got && c.lane == 0) c.release(ring, 1);
      }
      if (!per_slot) {
        const uint64_t tb = p.stamps ? global_ns() : 0;
        bar_sync(kBarConsumers, kNC * 32);  // h buffer b is free again
        if (p.stamps && c.tid == 0) c.count(ST_D_BAR_NS, global_ns() - tb);
        if (c.tid == 0) issue_ready(used + 1 + nbuf, false);
      }
      ++used;
      sl0 = sl1;
    }
    if (rb == nrb - 1 && c.tid == 0) c.stamp(ST_D_SUMMED);
    // Reduce each row's partial sums over the group's threads and write out.
    if (check_xflags && rb == 0) {
      if (!c.aborted()) wait_xflags(c);
      bar_sync(kBarConsumers, kNC * 32);
    }
    write_rows<FMT, MAXM>(c, acc, g, ch, active, nr, rb_lo);
  }
  // after an abort: h batches issued but not seen landing must land before exit
  if (c.tid == 0) {
    const uint64_t t = global_ns();
    for (int u = landed; u < issued; ++u) {
      while (!mbar_try_wait(hbar0 + 8u * (u % nbuf), (uint32_t)(u / nbuf) & 1u) && global_ns() - t < p.timeout_ns) {
      }
    }
  }
}

// --------------------------------------------------------------------------
// producer (lane 0 of the last warp issues; the warp stays converged)
// --------------------------------------------------------------------------
struct Producer {
  const Ctx& c;
  uint64_t pol;
  Ring ring;            // next stage to issue
  uint64_t used = 0;    // slots that received copies
  __device__ __forceinline__ Producer(const Ctx& cc) : c(cc) { pol = policy_evict_first(); }

  // Claims the next stage's slot and announces its bytes. False on abort.
  bool x_free = false;  // the consumers are done with x and the h area (down-phase slot in the x area)

  // Per-slot h fetches (single-kernel schedule, every pair fits the h area):
  // while it issues the down stages, the producer copies each slot's h values --
  // in pair order -- into the h area as soon as the slot's count is complete and
  // this CTA is done with the h area, counted on the slot's own mbarrier.
  const Route* h_rt = nullptr;  // set: fetches active
  int h_next = 0, h_nsl = 0;
  __device__ __forceinline__ bool test_x_free() {
    if (!x_free && mbar_test_wait(smem_u32(c.sm + c.p.off_xfree), 0)) x_free = true;
    return x_free;
  }
  __device__ __forceinline__ void poll_h() {
    const Params& p = c.p;
    if (!h_rt || h_next >= h_nsl || !test_x_free()) return;
    const float* rep = p.hbuf + (size_t)(blockIdx.x % kHRep) * p.npair_max * p.I;
    float* hs = reinterpret_cast<float*>(c.sm + p.off_hs);
    while (h_next < h_nsl && ld_relaxed_u32(p.ctrl + CTRL_SLOTCNT + h_next) >= (uint32_t)p.I) {
      __threadfence();             // acquire the slot's h stores ...
      fence_proxy_async_global();  // ... for the bulk copy that reads them
      const int p0 = h_rt->pair_base[h_next];
      const uint32_t bytes = (uint32_t)(h_rt->pair_base[h_next + 1] - p0) * (uint32_t)p.I * 4u;
      const uint32_t bar = c.full0 + 8u * (kHSlotBar + h_next);
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s_plain(smem_u32(hs + (size_t)p0 * p.I), rep + (size_t)p0 * p.I, bytes, bar);
      ++h_next;
    }
  }
  // Bounded: the remaining fetches once every down stage is issued.
  __device__ __forceinline__ void finish_h() {
    uint32_t spins = 0;
    while (h_rt && h_next < h_nsl && !c.aborted()) {
      poll_h();
      if (h_next >= h_nsl) break;
      __nanosleep(64);
      if ((++spins & 15) == 0) {
        if (c.peer_failed()) return;
        if (c.expired()) {
          c.fail(SITE_HIDDEN);
          return;
        }
      }
    }
  }
  // After an abort: the fetches issued must land before exit.
  __device__ __forceinline__ void drain_h() const {
    const uint64_t t = global_ns();
    for (int sl = 0; sl < h_next; ++sl)
      while (!mbar_try_wait(c.full0 + 8u * (kHSlotBar + sl), 0) && global_ns() - t < c.p.timeout_ns) {
      }
  }

  // Slot-interleaved schedule: a down stage carries the h rows of its slot
  // behind the weights. The producer copies the weights when it issues the
  // stage; the hand-off warp adds the h rows (counted on the same full barrier)
  // once every CTA has counted the slot's gate/up items as stored.
  // Gate/up stages of union slot s: this CTA's block of the slot's rows.
  __device__ __forceinline__ void ilv_pairs(const Route& rt, int s, int q) {
    const Params& p = c.p;
    int lo, hi;
    ilv_rows(p, s, lo, hi);
    const int e = s < p.S ? -1 - s : rt.slot_e[s];
    for (ItemWalk w(s * p.I + lo, s * p.I + hi, q, p.I); w.more(); ring.next(p.nslots)) {
      const int nq = w.count();
      uint32_t dst, bar;
      if (!begin((uint32_t)nq * p.pair_bytes + p.sc13e, dst, bar)) return;
      copy_pairs(e, w.j, nq, dst, bar);
      w.advance(nq);
    }
  }
  // The down stage of union slot s: this CTA's output rows of the expert's down
  // matrix now; the hand-off warp adds the slot's h rows later.
  __device__ __forceinline__ void ilv_down(const Route& rt, int s) {
    const Params& p = c.p;
    int r_lo, r_hi;
    cta_rows(p, r_lo, r_hi);
    const int nr = r_hi - r_lo;
    const int e = s < p.S ? -1 - s : rt.slot_e[s];
    const uint8_t* wt = e >= 0 ? p.w2 : p.sh_w2;
    const uint8_t* ws = e >= 0 ? p.w2_s : p.sh_w2_s;
    const size_t row0 = (size_t)(e >= 0 ? e : -1 - e) * p.H + r_lo;
    const uint32_t cb = (uint32_t)nr * p.row2, sb = (uint32_t)nr * p.sc2;
    const uint32_t hb = (uint32_t)(rt.pair_base[s + 1] - rt.pair_base[s]) * (uint32_t)p.I * 4u;
    uint32_t dst, bar;
    if (!begin(cb + sb + (uint32_t)p.sc2e + hb, dst, bar)) return;
    bulk_g2s(dst, wt + row0 * p.row2, cb, bar, pol);
    if (sb) bulk_g2s(dst + (uint32_t)p.d_rows_stage * p.row2, ws + row0 * p.sc2, sb, bar, pol);
    if (p.sc2e)  // FP8: the expert's down scales
      bulk_g2s(dst + (uint32_t)p.d_soff, ws + (size_t)(e >= 0 ? e : -1 - e) * p.sc2e, (uint32_t)p.sc2e, bar, pol);
    reinterpret_cast<volatile int*>(c.sm + p.off_dslot)[s] = ring.slot;
    __threadfence_block();  // the barrier's byte count and the slot before the count of issued stages
    reinterpret_cast<volatile int*>(c.sm + p.off_ucnt)[ILV_DISSUED] = s + 1;
    ring.next(p.nslots);
  }

  __device__ __forceinline__ bool begin(uint32_t bytes, uint32_t& dst, uint32_t& bar, bool d = false) {
    if (c.aborted()) return false;
    if (h_rt) {  // poll the h fetches while the slot is busy
      uint32_t spins = 0;
      // wake on the slot's release or after 200 ns to poll the h counts
      while (!mbar_try_wait_ns(c.empty0 + 8u * ring.slot, ring.phase() ^ 1u, 200u)) {
        poll_h();
        if ((++spins & 15) == 0) {
          if (c.aborted()) return false;
          if (c.expired()) {
            c.fail(SITE_RING_EMPTY);
            return false;
          }
        }
      }
    } else if (!c.wait_empty(ring)) {
      return false;
    }
    if (d && ring.slot >= c.p.nslots && !x_free) {
      if (!c.wait_bar(smem_u32(c.sm + c.p.off_xfree), 0, SITE_RING_EMPTY)) return false;
      x_free = true;
    }
    dst = smem_u32(c.slot_ptr(ring.slot, d));
    bar = c.full0 + 8u * ring.slot;
    c.slot_seq[ring.slot] = ring.seq;  // before arming: see Ctx::wait_full
    mbar_arrive_expect_tx(bar, bytes);
    used |= 1ull << ring.slot;
    return true;
  }

  // x rows straight into shared memory, ahead of any weights.
  __device__ __forceinline__ void x_rows() {
    const Params& p = c.p;
    const uint32_t bytes = (uint32_t)p.M * p.H * 2;
    mbar_arrive_expect_tx(c.xbar, bytes);
    bulk_g2s(smem_u32(c.sm + p.off_x), p.x, bytes, c.xbar, pol);
  }

  __device__ __forceinline__ void router() {
    const Params& p = c.p;
    int lo, hi;
    split_range(p.E / 2, blockIdx.x, p.grid, lo, hi);
    ring.fit(p.nslots);
    for (ItemWalk w(lo, hi, p.qr, 0); w.more(); ring.next(p.nslots)) {
      const int nq = w.count();
      const uint32_t bytes = (uint32_t)nq * p.rpair_bytes;
      uint32_t dst, bar;
      if (!begin(bytes, dst, bar)) return;
      // several smaller copies: each bulk copy streams at a fraction of the SM's
      // bandwidth, and the router rows are on the critical path
      const uint8_t* src = p.router_w + (size_t)w.a * p.rpair_bytes;
      for (uint32_t o = 0; o < bytes; o += kRouterCopy) {
        const uint32_t nb = min((uint32_t)kRouterCopy, bytes - o);
        bulk_g2s(dst + o, src + o, nb, bar, pol);
      }
      w.advance(nq);
    }
  }

  // Rows j .. j + nq - 1 of expert e (shared expert -1 - e when e < 0) as a
  // gate block and an up block (plus the two scale blocks for NVFP4).
  __device__ __forceinline__ void copy_pairs(int e, int j, int nq, uint32_t dst, uint32_t bar) const {
    const Params& p = c.p;
    const uint8_t* wt = e >= 0 ? p.w13 : p.sh_w13;
    const uint8_t* ws = e >= 0 ? p.w13_s : p.sh_w13_s;
    const size_t ex = (size_t)(e >= 0 ? e : -1 - e);
    const size_t rg = ex * 2 * p.I + j, ru = rg + p.I;  // first gate row, first up row
    const uint32_t cb = (uint32_t)nq * p.row13;
    bulk_g2s(dst, wt + rg * p.row13, cb, bar, pol);
    bulk_g2s(dst + cb, wt + ru * p.row13, cb, bar, pol);
    if (p.sc13e) bulk_g2s(dst + 2 * cb, ws + ex * p.sc13e, (uint32_t)p.sc13e, bar, pol);  // FP8: the expert's scales
    if (p.sc13) {
      const uint32_t sb = (uint32_t)nq * p.sc13;
      bulk_g2s(dst + 2 * cb, ws + rg * p.sc13, sb, bar, pol);
      bulk_g2s(dst + 2 * cb + sb, ws + ru * p.sc13, sb, bar, pol);
    }
  }

  // Gate/up stages: consecutive rows of one expert as a gate block and an up
  // block (plus the two scale blocks for NVFP4).
  // q: items per stage (0: the planned stage size).
  __device__ __forceinline__ void pairs(bool shared_phase, const Route& rt, int q = 0) {
    const Params& p = c.p;
    int lo, hi;
    if (shared_phase) {
      split_range(p.S * p.I, blockIdx.x, p.grid, lo, hi);
    } else {
      lo = c.misc[MISC_ULO];
      hi = c.misc[MISC_UHI];
    }
    const int nsl_ring = shared_phase ? p.nslots : p.nslots + p.nslots_x;
    ring.fit(nsl_ring);
    for (ItemWalk w(lo, hi, q > 0 ? q : p.q, p.I); w.more(); ring.next(nsl_ring)) {
      const int nq = w.count();
      const int slot = w.u + (shared_phase ? 0 : p.S);
      uint32_t dst, bar;
      if (!begin((uint32_t)nq * p.pair_bytes + p.sc13e, dst, bar)) return;
      copy_pairs(shared_phase ? -1 - slot : rt.slot_e[slot], w.j, nq, dst, bar);
      w.advance(nq);
    }
  }

  // Down stages (row block rb, union slot sl) for sl in [sl_lo, sl_hi).
  // nd: down-phase slots in the x area (0 or 1)
  __device__ __forceinline__ void down_block(const Route& rt, int rb, int sl_lo, int sl_hi, int nd) {
    const Params& p = c.p;
    int r_lo, r_hi;
    cta_rows(p, r_lo, r_hi);
    const int rb_lo = r_lo + rb * p.d_rows_stage;
    const int nr = min(p.d_rows_stage, r_hi - rb_lo);
    ring.fit(p.nslots + nd);
    for (int sl = sl_lo; sl < sl_hi; ++sl) {
      const int e = sl < p.S ? -1 - sl : rt.slot_e[sl];
      const uint8_t* wt = e >= 0 ? p.w2 : p.sh_w2;
      const uint8_t* ws = e >= 0 ? p.w2_s : p.sh_w2_s;
      const size_t ex = (size_t)(e >= 0 ? e : -1 - e);
      const size_t row0 = ex * p.H + rb_lo;
      const uint32_t cb = (uint32_t)nr * p.row2, sb = (uint32_t)nr * p.sc2;
      uint32_t dst, bar;
      if (!begin(cb + sb + (uint32_t)p.sc2e, dst, bar, true)) return;
      bulk_g2s(dst, wt + row0 * p.row2, cb, bar, pol);
      if (sb) bulk_g2s(dst + (uint32_t)p.d_rows_stage * p.row2, ws + row0 * p.sc2, sb, bar, pol);
      if (p.sc2e) bulk_g2s(dst + (uint32_t)p.d_soff, ws + ex * p.sc2e, (uint32_t)p.sc2e, bar, pol);  // FP8 scales
      ring.next(p.nslots + nd);
    }
  }

  __device__ __forceinline__ int down_blocks() const {
    int r_lo, r_hi;
    cta_rows(c.p, r_lo, r_hi);
    return (r_hi - r_lo + c.p.d_rows_stage - 1) / c.p.d_rows_stage;
  }

  // Speculative expert prefetch ("Muse Spark Open Ultrafast", section
  // "Speculative expert prefetching": consecutive steps tend to route alike, so
  // the experts the previous step used most are pulled into L2 while the router
  // runs and HBM is otherwise idle). This CTA's 1/grid share of every byte of
  // each listed expert (gate/up and down codes and scales) into L2; the list is
  // the one the previous run of this handle left for this run's parity.
  // Issued in 16 KB pieces, one at a time and only until the routing warps flag
  // the routing as done: the CTA's bulk-copy unit handles its operations in
  // order, and a long prefetch queued ahead of the routed stages would delay them.
  __device__ __forceinline__ void prefetch_predicted() const {
    const Params& p = c.p;
    if (p.pf_n <= 0 || p.hist == nullptr) return;
    const volatile int* routed = reinterpret_cast<const volatile int*>(c.misc) + MISC_ROUTED;
    const uint32_t ep = ld_relaxed_u32(&p.ctrl[CTRL_EPOCH]);
    const int* list = p.hist + (size_t)(ep & 1u) * kPfMax;
    const size_t n13 = (size_t)2 * p.I, n2 = (size_t)p.H;  // rows per expert (transposed down: same bytes)
    constexpr uint32_t kPiece = 16384;
    for (int i = 0; i < p.pf_n && i < kPfMax; ++i) {
      const int e = list[i];
      if (e < 0 || e >= p.E) continue;
      const uint8_t* base[4] = {p.w13 + (size_t)e * n13 * p.row13, p.w2 + (size_t)e * n2 * p.row2,
                                p.sc13 ? p.w13_s + (size_t)e * n13 * p.sc13 : nullptr,
                                p.sc2 ? p.w2_s + (size_t)e * n2 * p.sc2 : nullptr};
      const size_t len[4] = {n13 * p.row13, n2 * p.row2, n13 * p.sc13, n2 * p.sc2};
      for (int r = 0; r < 4; ++r) {
        if (!base[r]) continue;
        int lo, hi;  // 16-byte units of this CTA's share
        split_range((int)(len[r] / 16), blockIdx.x, p.grid, lo, hi);
        for (size_t o = (size_t)lo * 16; o < (size_t)hi * 16; o += kPiece) {
          if (*routed || c.aborted()) return;
          const uint32_t n = (uint32_t)min((size_t)kPiece, (size_t)hi * 16 - o);
          bulk_prefetch_l2(base[r] + o, n);
          __nanosleep(200);
        }
      }
    }
  }

  // Shared experts' down rows of this CTA into L2 ahead of time.
  __device__ __forceinline__ void prefetch_shared_down() {
    const Params& p = c.p;
    int r_lo, r_hi;
    cta_rows(p, r_lo, r_hi);
    if (r_hi <= r_lo) return;
    for (int s = 0; s < p.S; ++s) {
      const size_t row0 = (size_t)s * p.H + r_lo;
      bulk_prefetch_l2(p.sh_w2 + row0 * p.row2, (uint32_t)(r_hi - r_lo) * p.row2);
      if (p.sc2) bulk_prefetch_l2(p.sh_w2_s + row0 * p.sc2, (uint32_t)(r_hi - r_lo) * p.sc2);
    }
  }

  // Before exit: wait (bounded) for this CTA's copies still in flight: the
  // newest use of every slot that received copies.
  __device__ __forceinline__ void drain() {
    const Params& p = c.p;
    const uint64_t t = global_ns();
    for (uint64_t u = used; u; u &= u - 1) {
      const int s = __ffsll((long long)u) - 1;
      const uint32_t bar = c.full0 + 8u * (uint32_t)s;
      const uint32_t par = (uint32_t)((ring.par >> s) & 1u) ^ 1u;  // the parity of its last use
      while (!mbar_try_wait(bar, par)) {
        if (global_ns() - t > p.timeout_ns) {
          c.fail(SITE_DRAIN);
          return;
        }
      }
    }
  }
};

// --------------------------------------------------------------------------
// the kernel: PHASES = PH_ALL (single persistent kernel) or one phase group of
// the three-kernel chain (PH_R, PH_U, PH_D).
// --------------------------------------------------------------------------
template <int FMT, int MAXM, int PHASES>
__global__ void __launch_bounds__(kThreads, 1) moe_layer_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctx c(p, sm);
  Route rt(p, sm);
  constexpr bool kChain = PHASES != PH_ALL;
  constexpr bool kNeedX = (PHASES & (PH_R | PH_U)) != 0;
  constexpr bool kRoute = (PHASES & (PH_U | PH_D)) != 0;
  constexpr bool kLast = (PHASES & PH_D) != 0;

  if (kChain) pdl_launch_dependents();
  if (c.tid == 0) {
    for (int i = 0; i < p.nslots + max(p.nslots_x, p.nslots_d); ++i) {
      mbar_init(c.full0 + 8u * i, 1);
      mbar_init(c.empty0 + 8u * i, kNC);
      c.slot_seq[i] = -1;
    }
    mbar_init(c.xbar, 1);
    mbar_init(smem_u32(sm + p.off_xfree), 1);
    if (PHASES == PH_ALL && p.hs_perslot)
      for (int i = 0; i < p.nslot_max; ++i) mbar_init(c.full0 + 8u * (kHSlotBar + i), 1);
    mbar_init(smem_u32(sm + p.off_hbar), 1);
    mbar_init(smem_u32(sm + p.off_hbar) + 8u, 1);
    mbar_init_fence();
    c.misc[MISC_ABORT] = 0;
    c.misc[MISC_NROUTED] = 0;
    c.misc[MISC_ROUTED] = 0;
  }
  for (int e = c.tid; e < p.E; e += kThreads) rt.emask[e] = 0u;
  for (int e = c.tid; e < (p.E + 31) / 32; e += kThreads) rt.bitmap[e] = 0u;
  __syncthreads();

  bool x_issued = false;
  if (c.warp < kNC) {
    // ------------------------------------------------------------ consumers
    if (kChain) pdl_wait();
    if (c.tid == 0) c.misc[MISC_EPOCH] = (int)ld_relaxed_u32(&p.ctrl[CTRL_EPOCH]);
    if (kNeedX) prepare_x(c, FMT != FMT_BF16);
    bar_sync(kBarConsumers, kNC * 32);
    if (c.tid == 0) c.stamp(ST_X_LOADED);
    if (PHASES == PH_ALL && p.out_aliases_x && c.tid == 0)
      st_tagged(p.xflags + blockIdx.x, c.epoch(), 0.0f);
    Ring ring;
    if constexpr (PHASES == PH_ALL) {
      // Every warp computes this CTA's router rows; then warps 0 .. nrw - 1
      // route while the others compute the shared experts' gate/up items.
      ring = consume_router<MAXM>(c, ring);
      bar_sync(kBarConsumers, kNC * 32);  // this CTA's logits are all stored
      if (c.tid == 0) {
        c.stamp(ST_RFLAG);
      }
      if (FMT != FMT_BF16) {  // the router is done with the bf16 x rows
        x_to_f16(c);
        bar_sync(kBarConsumers, kNC * 32);
      }
      const int nrw = ilv_nrw(p);
      if (c.warp < nrw) {
        route_rows<MAXM>(c, rt, true, nrw * 32, kBarRouting);
        if (c.tid == 0) reinterpret_cast<volatile int*>(c.misc)[MISC_ROUTED] = 1;  // hint for the producer's prefetch
        bar_arrive(kBarRoute, (nrw + 1) * 32);
        if (c.tid == 0) c.stamp(ST_ROUTED);
      }
      ring = consume_items<FMT, MAXM>(c, rt, ITEM_SHARED, ring, nrw, ilv_snw(p), ilv_sq(p));
      fence_proxy_async_global();  // the h stores are read by other CTAs' bulk copies
      bar_sync(kBarConsumers, kNC * 32);  // the routing tables, and this CTA's shared h rows all stored
      if (c.tid == 0) {
        c.stamp(ST_R_DONE);
        if (p.S > 0 && p.hs_nbuf == 2) {
          __threadfence();  // release them with the count
          count_done(p, CTRL_SCOUNT);
        }
      }
      ring = consume_items<FMT, MAXM>(c, rt, ITEM_ROUTED, ring);
      fence_proxy_async_global();
      if (c.tid == 0) c.stamp(ST_U_DONE);
    } else {
      if (PHASES & PH_R) {
        ring = consume_router<MAXM>(c, ring);
        bar_sync(kBarConsumers, kNC * 32);  // this CTA's logits are all stored
        if (c.tid == 0) {
          c.stamp(ST_RFLAG);
        }
      }
      if (kRoute) {
        route_rows<MAXM>(c, rt, (PHASES & PH_U) != 0);
        if (c.tid == 0) reinterpret_cast<volatile int*>(c.misc)[MISC_ROUTED] = 1;  // hint for the producer's prefetch
        bar_arrive(kBarRoute, kThreads);
        if (c.tid == 0) c.stamp(ST_ROUTED);
      }
      if (FMT != FMT_BF16 && kNeedX) {  // the router is done with the bf16 x rows
        x_to_f16(c);
        bar_sync(kBarConsumers, kNC * 32);
      }
      // gate/up items: the shared experts' (their stages were issued before
      // routing), then the routed experts'; one loop so that the code exists once
      constexpr int kKind0 = (PHASES & PH_R) ? ITEM_SHARED : ITEM_ROUTED;
      constexpr int kKind1 = (PHASES & PH_U) ? ITEM_ROUTED : ITEM_SHARED;
      if (PHASES & (PH_R | PH_U)) {
#pragma unroll 1
        for (int kind = kKind0; kind <= kKind1; ++kind) {
          ring = consume_items<FMT, MAXM>(c, rt, kind, ring);
          fence_proxy_async_global();  // the h stores are read by other CTAs' bulk copies
          if (c.tid == 0) c.stamp(kind == ITEM_SHARED ? ST_R_DONE : ST_U_DONE);
        }
      }
    }
    if (PHASES & PH_U) {
      // the h area takes bulk copies from here on (per-slot h fetches)
      if (PHASES == PH_ALL && p.hs_perslot) fence_proxy_async_shared();
      bar_sync(kBarConsumers, kNC * 32);  // this CTA's h rows are all stored
      if (c.tid == 0) {
        __threadfence();  // release them with the count(s)
        count_done(p, CTRL_UCOUNT);
        if (PHASES == PH_ALL && p.hs_perslot) count_slots(c);
        if (PHASES == PH_ALL) mbar_arrive(smem_u32(sm + p.off_xfree), 1);  // x and the h area are free
      }
    }
    if (PHASES & PH_D)
      consume_down<FMT, MAXM>(c, rt, PHASES == PH_ALL && p.out_aliases_x, PHASES == PH_ALL, ring,
                              PHASES == PH_ALL ? p.nslots_d : 0);
    if (kLast) write_prediction(c, rt);
    if (c.tid == 0) {
      c.stamp(ST_D_DONE);
      if (p.stamps) {
        p.stamps[(size_t)blockIdx.x * kStampSlots + ST_CLOCK_MHZ] =
            (unsigned long long)(clock64() - c.c0) * 1000ull / (global_ns() - c.t0 + 1);
      }
    }
  } else {
    // ------------------------------------------------------------ producer
    Producer pr(c);
    if (c.lane == 0) {
      c.stamp(ST_START);
      if (PHASES == PH_ALL) {
        pr.x_rows();
        x_issued = true;
      }
      if (PHASES & PH_R) pr.router();
      if (kChain && kNeedX) {
        pdl_wait();  // x may be the previous kernel's output
        if (!c.aborted()) {
          pr.x_rows();
          x_issued = true;
        }
      }
      if (PHASES & PH_R) {
        // single kernel: the shared stages are sized for the warps that do not route
        pr.pairs(true, rt, PHASES == PH_ALL ? ilv_sq(p) : 0);
        c.stamp(ST_P_R_ISSUED);
        if (PHASES & PH_D) pr.prefetch_shared_down();
        pr.prefetch_predicted();
      } else if (PHASES == PH_D) {
        // The shared experts' down rows of the first row block need no routing.
        if (pr.down_blocks() > 0) pr.down_block(rt, 0, 0, p.S, 0);
      }
    }
    if (kRoute) {
      __syncwarp();
      bar_sync(kBarRoute, PHASES == PH_ALL ? (ilv_nrw(p) + 1) * 32 : kThreads);
    }
    if (c.lane == 0) {
      c.stamp(ST_P_ROUTE);
      if (PHASES & PH_U) {
        pr.pairs(false, rt);
        c.stamp(ST_P_U_ISSUED);
      }
      if (PHASES & PH_D) {
        const int nsl = p.S + c.misc[MISC_NROUTED];
        const int first = PHASES == PH_D ? p.S : 0;  // the chain issued these before routing
        const int nd = PHASES == PH_ALL ? p.nslots_d : 0;
        if (PHASES == PH_ALL && p.hs_perslot) {
          pr.h_rt = &rt;
          pr.h_nsl = nsl;
        }
        for (int rb = 0; rb < pr.down_blocks(); ++rb) pr.down_block(rt, rb, rb == 0 ? first : 0, nsl, nd);
        pr.finish_h();
        c.stamp(ST_P_D_ISSUED);
      }
      if (c.aborted()) {
        pr.drain();
        pr.drain_h();
      }
      // the x copy may still be in flight if the consumers gave up before it landed
      if (x_issued && c.aborted()) {
        const uint64_t t = global_ns();
        while (!mbar_try_wait(c.xbar, 0) && global_ns() - t < p.timeout_ns) {
        }
      }
    }
    __syncwarp();
  }
  __syncthreads();
  if (kLast && c.tid == 0) {
    const uint32_t prev = atomicAdd(&p.ctrl[CTRL_EXIT], 1u);
    if (prev == gridDim.x - 1) {
      p.ctrl[CTRL_EXIT] = 0u;
      *reinterpret_cast<unsigned long long*>(p.ctrl + CTRL_UCOUNT) = 0ull;
      *reinterpret_cast<unsigned long long*>(p.ctrl + CTRL_SCOUNT) = 0ull;
      if (PHASES == PH_ALL && p.hs_perslot)
        for (int i = 0; i < p.nslot_max; ++i) p.ctrl[CTRL_SLOTCNT + i] = 0u;
      uint32_t e = p.ctrl[CTRL_EPOCH] + 1u;
      if (e == 0xffffffffu) e = 0u;
      p.ctrl[CTRL_EPOCH] = e;
    }
  }
}

// --------------------------------------------------------------------------
// the slot-interleaved single kernel
// --------------------------------------------------------------------------
// Gate/up items of union slot s (this CTA's row block), then the warp's arrival
// on the slot's counter in shared memory (a CTA-scope release of its h stores).
template <int FMT, int MAXM>
__device__ __forceinline__ Ring ilv_items(const Ctx& c, const Route& rt, int s, Ring ring, int& rot, int w0, int nw,
                                          int q) {
  const Params& p = c.p;
  int lo, hi;
  ilv_rows(p, s, lo, hi);
  if (hi > lo) {
    const uint4* xs = reinterpret_cast<const uint4*>(c.sm + p.off_x);
    XRegs<FMT, MAXM> xr;
    load_xregs<FMT, MAXM>(c, xr);
    ItemWalk w(s * p.I + lo, s * p.I + hi, q, p.I);
    w.w0 = w0;
    w.nw = nw;
    w.r = rot;  // the warp rotation carries over between slots
    for (; w.more(); ring.next(p.nslots)) {
      item_stage<FMT, MAXM>(c, rt, w, ring, s, s < p.S, xr, xs, false);
      w.advance(w.count());
    }
    rot = w.r;
    fence_proxy_async_global();  // the h stores are read by other CTAs' bulk copies
  }
  // arrival (every warp, every slot, with or without items): the hand-off warp
  // counts the slot done when all kNC warps have arrived
  __syncwarp();
  if (c.lane == 0) {
    __threadfence_block();
    atomicAdd(reinterpret_cast<int*>(c.sm + p.off_ucnt) + (s & (kIlvCnt - 1)), 1);
  }
  return ring;
}

// The down stage of union slot s: the CTA's output rows of the expert's down
// matrix against the slot's h rows, both in the stage's ring slot.
template <int FMT, int MAXM>
__device__ __forceinline__ Ring ilv_down(const Ctx& c, const Route& rt, int s, Ring ring,
                                         float (&acc)[rows_per_group(FMT)][MAXM], int g, int ch, bool active,
                                         int nr, int r_lo) {
  const Params& p = c.p;
  const bool got = !c.aborted() && c.wait_full(ring);
  if (got && active) {
    const uint8_t* st = c.slot_ptr(ring.slot);
    down_stage<FMT, MAXM>(p, st, reinterpret_cast<const float*>(st + p.d_hoff), rt.slot_mask[s], acc, g, ch, nr,
                          fp8_down_scales(c, ring, false, s < p.S ? -1 - s : rt.slot_e[s]), r_lo);
  }
  __syncwarp();
  if (got && c.lane == 0) c.release(ring, 1);
  ring.next(p.nslots);
  return ring;
}

// The h rows of slot s into its down stage's ring slot (hand-off warp, lane 0).
__device__ __forceinline__ void ilv_fetch(const Ctx& c, const Route& rt, int s) {
  const Params& p = c.p;
  const int rs = reinterpret_cast<const volatile int*>(c.sm + p.off_dslot)[s];
  const int p0 = rt.pair_base[s];
  const uint32_t bytes = (uint32_t)(rt.pair_base[s + 1] - p0) * (uint32_t)p.I * 4u;
  const float* src = p.hbuf + ((size_t)(blockIdx.x % kHRep) * p.npair_max + p0) * p.I;
  fence_proxy_async_global();  // the acquired h stores before the bulk copy that reads them
  bulk_g2s_plain(smem_u32(c.slot_ptr(rs) + p.d_hoff), src, bytes, c.full0 + 8u * (uint32_t)rs);
}

// Two hand-off warps keep GPU-scope fences and L2 polls away from the consumer
// warps and the producer. The publisher (lane 0) counts this CTA's gate/up
// items of a slot as stored once every consumer warp has arrived, with one fence
// for all slots found complete.
__device__ __forceinline__ void ilv_publish(const Ctx& c) {
  const Params& p = c.p;
  volatile int* w = reinterpret_cast<volatile int*>(c.sm + p.off_ucnt);
  const int nsl = p.S + c.misc[MISC_NROUTED];
  uint32_t spins = 0;
  for (int pub = 0; pub < nsl;) {
    int np = pub;
    while (np < nsl && w[np & (kIlvCnt - 1)] >= kNC * (np / kIlvCnt + 1)) ++np;
    if (np > pub) {
      __threadfence();  // acquires the warps' h stores (through the counters) and releases them
      for (; pub < np; ++pub) {
        int lo, hi;
        ilv_rows(p, pub, lo, hi);
        if (hi > lo) red_add_u32(p.ctrl + CTRL_SLOTCNT + pub, (uint32_t)(hi - lo));
      }
      continue;
    }
    __nanosleep(32);
    // the consumers arrive even after an abort; bounded all the same
    if ((++spins & 63) == 0 && global_ns() - c.t0 > 2 * p.timeout_ns) {
      c.fail(SITE_HIDDEN);
      return;
    }
  }
}

// The fetcher (lane 0) copies the h rows of each issued down stage once every
// CTA has counted the slot. After an abort it copies the remaining h parts
// anyway, so that every armed full barrier completes.
__device__ __forceinline__ void ilv_fetcher(const Ctx& c, const Route& rt) {
  const Params& p = c.p;
  volatile int* w = reinterpret_cast<volatile int*>(c.sm + p.off_ucnt);
  int hn = 0;
  uint32_t spins = 0;
  bool failed = false;
  for (;;) {
    const int di = w[ILV_DISSUED];
    __threadfence_block();  // the issued stages' slots after their count
    const bool ab = c.aborted();
    bool progress = false;
    while (hn < di && (ab || ld_acquire_u32(p.ctrl + CTRL_SLOTCNT + hn) >= (uint32_t)p.I)) {
      ilv_fetch(c, rt, hn++);
      progress = true;
    }
    if (w[ILV_PDONE] && hn == w[ILV_DISSUED]) break;
    if (!progress) {
      __nanosleep(32);
      if ((++spins & 15) == 0) {
        if (!ab && c.peer_failed()) c.abort_local();  // another CTA gave up: stop waiting on it
        if (c.expired()) {
          if (!failed) c.fail(SITE_HIDDEN);
          failed = true;
          if (global_ns() - c.t0 > 2 * p.timeout_ns) break;  // bounded even if the others stall
        }
      }
    }
  }
}

// One kernel for the whole step, phases overlapped slot by slot: router rows
// and the shared experts' gate/up rows, routing, then for t = S, S + 1, ...:
// the gate/up items of slot t and every down stage of a slot s with
// s + lag <= t. A down stage needs the h rows of its slot from every CTA; the
// lag leaves the slot's count time to complete while later gate/up stages stream.
template <int FMT, int MAXM>
__global__ void __launch_bounds__(kThreadsIlv, 1) moe_ilv_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctx c(p, sm);
  Route rt(p, sm);
  if (c.tid == 0) {
    for (int i = 0; i < p.nslots; ++i) {
      mbar_init(c.full0 + 8u * i, 1);
      mbar_init(c.empty0 + 8u * i, kNC);
      c.slot_seq[i] = -1;
    }
    mbar_init(c.xbar, 1);
    mbar_init_fence();
    c.misc[MISC_ABORT] = 0;
    c.misc[MISC_NROUTED] = 0;
    c.misc[MISC_ROUTED] = 0;
  }
  if (c.tid < ILV_WORDS) reinterpret_cast<int*>(sm + p.off_ucnt)[c.tid] = 0;
  for (int e = c.tid; e < p.E; e += kThreadsIlv) rt.emask[e] = 0u;
  for (int e = c.tid; e < (p.E + 31) / 32; e += kThreadsIlv) rt.bitmap[e] = 0u;
  __syncthreads();

  int r_lo, r_hi;
  cta_rows(p, r_lo, r_hi);
  const int nr = r_hi - r_lo;  // every output row of the CTA in one down stage (planned)
  if (c.warp < kNC) {
    // ------------------------------------------------------------ consumers
    if (c.tid == 0) c.misc[MISC_EPOCH] = (int)ld_relaxed_u32(&p.ctrl[CTRL_EPOCH]);
    prepare_x(c, FMT != FMT_BF16);
    bar_sync(kBarConsumers, kNC * 32);
    if (c.tid == 0) c.stamp(ST_X_LOADED);
    if (p.out_aliases_x && c.tid == 0) st_tagged(p.xflags + blockIdx.x, c.epoch(), 0.0f);
    Ring ring;
    ring = consume_router<MAXM>(c, ring);
    bar_sync(kBarConsumers, kNC * 32);  // this CTA's logits are all stored
    if (c.tid == 0) {
      c.stamp(ST_RFLAG);
    }
    if (FMT != FMT_BF16) {  // the router is done with the bf16 x rows
      x_to_f16(c);
      bar_sync(kBarConsumers, kNC * 32);
    }
    const int nrw = ilv_nrw(p);
    if (c.warp < nrw) {
      route_rows<MAXM>(c, rt, true, nrw * 32, kBarRouting);
      if (c.tid == 0) reinterpret_cast<volatile int*>(c.misc)[MISC_ROUTED] = 1;  // hint for the producer's prefetch
      bar_arrive(kBarRoute, ilv_route_threads(p));
      if (c.tid == 0) c.stamp(ST_ROUTED);
    }
    constexpr int RPG = rows_per_group(FMT);
    const int g = c.tid / p.tg, ch = c.tid % p.tg;
    const bool active = g < p.ng;
    float acc[RPG][MAXM];
#pragma unroll
    for (int ri = 0; ri < RPG; ++ri)
#pragma unroll
      for (int m = 0; m < MAXM; ++m) acc[ri][m] = 0.0f;
    int rot = 0, dnext = 0;
    // the shared experts' items: the non-routing warps compute them while routing
    // runs; the routing warps walk the same stages (without items) afterwards
#pragma unroll 1
    for (int s = 0; s < p.S; ++s) ring = ilv_items<FMT, MAXM>(c, rt, s, ring, rot, nrw, ilv_snw(p), ilv_sq(p));
    bar_sync(kBarConsumers, kNC * 32);  // the routing tables, for every warp
    if (c.tid == 0) c.stamp(ST_R_DONE);
    const int nsl = p.S + c.misc[MISC_NROUTED];
    rot = 0;
#pragma unroll 1
    for (int t = p.S; t < nsl + p.ilv_lag; ++t) {
      if (t < nsl) ring = ilv_items<FMT, MAXM>(c, rt, t, ring, rot, 0, kNC, p.q);
      while (nr > 0 && dnext < nsl && dnext + p.ilv_lag <= t)
        ring = ilv_down<FMT, MAXM>(c, rt, dnext++, ring, acc, g, ch, active, nr, r_lo);
    }
    if (c.tid == 0) c.stamp(ST_D_SUMMED);
    if (nr > 0) {
      if (p.out_aliases_x) {
        if (!c.aborted()) wait_xflags(c);
        bar_sync(kBarConsumers, kNC * 32);
      }
      write_rows<FMT, MAXM>(c, acc, g, ch, active, nr, r_lo);
    }
    write_prediction(c, rt);
    if (c.tid == 0) {
      c.stamp(ST_D_DONE);
      if (p.stamps) {
        p.stamps[(size_t)blockIdx.x * kStampSlots + ST_CLOCK_MHZ] =
            (unsigned long long)(clock64() - c.c0) * 1000ull / (global_ns() - c.t0 + 1);
      }
    }
  } else if (c.warp == kNC) {
    // ------------------------------------------------------------ producer
    Producer pr(c);
    if (c.lane == 0) {
      c.stamp(ST_START);
      pr.x_rows();
      pr.router();
      for (int s = 0; s < p.S; ++s) pr.ilv_pairs(rt, s, ilv_sq(p));
      c.stamp(ST_P_R_ISSUED);
      pr.prefetch_shared_down();
      pr.prefetch_predicted();
    }
    __syncwarp();
    bar_sync(kBarRoute, ilv_route_threads(p));
    if (c.lane == 0) {
      c.stamp(ST_P_ROUTE);
      const int nsl = p.S + c.misc[MISC_NROUTED];
      int dnext = 0;
      for (int t = p.S; t < nsl + p.ilv_lag; ++t) {
        if (t < nsl) pr.ilv_pairs(rt, t, p.q);
        while (nr > 0 && dnext < nsl && dnext + p.ilv_lag <= t) pr.ilv_down(rt, dnext++);
      }
      c.stamp(ST_P_D_ISSUED);
      __threadfence_block();
      reinterpret_cast<volatile int*>(sm + p.off_ucnt)[ILV_PDONE] = 1;
      if (c.aborted()) {
        pr.drain();  // the hand-off warp completes the h parts of armed down stages
        // the x copy may still be in flight if the consumers gave up before it landed
        const uint64_t t = global_ns();
        while (!mbar_try_wait(c.xbar, 0) && global_ns() - t < p.timeout_ns) {
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ hand-off warps
    __syncwarp();
    bar_sync(kBarRoute, ilv_route_threads(p));
    if (c.lane == 0) {
      if (c.warp == kNC + 1)
        ilv_publish(c);
      else
        ilv_fetcher(c, rt);
    }
    __syncwarp();
  }
  __syncthreads();
  if (c.tid == 0) {
    const uint32_t prev = atomicAdd(&p.ctrl[CTRL_EXIT], 1u);
    if (prev == gridDim.x - 1) {
      p.ctrl[CTRL_EXIT] = 0u;
      for (int i = 0; i < p.nslot_max; ++i) p.ctrl[CTRL_SLOTCNT + i] = 0u;
      uint32_t e = p.ctrl[CTRL_EPOCH] + 1u;
      if (e == 0xffffffffu) e = 0u;
      p.ctrl[CTRL_EPOCH] = e;
    }
  }
}

}  // namespace moe
