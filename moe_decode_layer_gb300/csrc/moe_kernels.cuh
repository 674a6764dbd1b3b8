// Kernels of the small-batch MoE decode layer step (sm_103a).
//
// Every CTA has kNC consumer warps and one producer warp. The producer streams
// weight rows from HBM into a ring of shared-memory slots with 1-D bulk (TMA)
// copies tagged evict-first in L2, each slot guarded by a "full" mbarrier (the
// copy engine counts the bytes in) and an "empty" mbarrier (consumers hand the
// slot back). Consumers turn slots into dot products against the token rows.
//
// Phases (Ling-3.0-flash batch-1 decode blog, section "PDL: stacking the latency
// floors of small kernels": router chain norm -> gate matvec -> top-k, MoE chain
// up-GEMM -> activation -> down-GEMM -> combine):
//   R  router rows (bf16) and the shared experts' gate/up rows: router logits and
//      the shared experts' silu(g) * u; both need no routing decision.
//   T  every CTA reads all logits and selects the top-k of each row itself, then
//      forms the union of chosen experts with one row bitmask per expert and a
//      popcount prefix over the expert ids (SGLang Low-Latency Mode page,
//      section "Low-Latency-Specific Optimizations", item 3).
//   U  gate/up rows of the chosen experts: h = w * silu(g) * u per (expert, row);
//      SwiGLU in fp32 right after the dot products (blog section "Two fusions and
//      a retune").
//   D  down rows: each CTA owns a contiguous block of output features, sums
//      W2_e h_e over all chosen and shared experts in fp32 and writes
//      bf16(residual + sum) with one rounding (blog section "PDL: ...": the combine
//      is an fp32 sum with a single final cast).
//
// Hand-offs between CTAs carry no fence and no flag: every value is stored as a
// 64-bit word (run tag << 32 | fp32 bits) and readers poll until the tag equals
// the current run's tag ("Muse Spark Open Ultrafast", section "Megakernel
// internals", part 3: a GPU-scope fence with bulk loads in flight costs
// microseconds, so the data carries its own readiness). The tag is a per-handle
// counter that the last CTA of a run advances, so buffers are never reset.
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

// --------------------------------------------------------------------------
// small helpers
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// [lo, hi) share of n items for CTA c of g.
__device__ __forceinline__ void split_range(long long n, int c, int g, long long& lo, long long& hi) {
  lo = n * c / g;
  hi = n * (c + 1) / g;
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

struct Ctx {
  const Params& p;
  uint8_t* sm;
  int* misc;
  volatile int* slot_seq;  // [nslots] ring stage that currently owns each slot
  uint32_t full0, empty0;
  uint64_t t0;
  int tid, warp, lane;

  __device__ Ctx(const Params& pp, uint8_t* base) : p(pp), sm(base) {
    misc = reinterpret_cast<int*>(sm + p.off_misc);
    slot_seq = reinterpret_cast<volatile int*>(sm + p.off_slot_seq);
    full0 = smem_u32(sm + p.off_full);
    empty0 = smem_u32(sm + p.off_empty);
    t0 = global_ns();
    tid = threadIdx.x;
    warp = tid >> 5;
    lane = tid & 31;
  }
  __device__ bool aborted() const { return *reinterpret_cast<volatile int*>(misc + MISC_ABORT) != 0; }
  __device__ void fail(uint32_t site) const {
    *reinterpret_cast<volatile int*>(misc + MISC_ABORT) = 1;
    atomicOr(&p.ctrl[CTRL_STATUS], DEV_ERR_TIMEOUT);
    atomicCAS(&p.ctrl[CTRL_WHERE], 0u, site);
  }
  __device__ bool expired() const { return global_ns() - t0 > p.timeout_ns; }
  // Another CTA gave up: stop waiting on data it will never publish.
  __device__ bool peer_failed() const { return ld_relaxed_u32(&p.ctrl[CTRL_STATUS]) != 0; }
  __device__ uint32_t epoch() const { return static_cast<uint32_t>(misc[MISC_EPOCH]); }
  __device__ uint8_t* slot_ptr(int slot) const { return sm + p.off_ring + (size_t)slot * p.slot_bytes; }
  // Phase timestamp (one plain store; off unless the handle has a stamp buffer).
  __device__ void stamp(int ev) const {
    if (p.stamps) p.stamps[(size_t)blockIdx.x * kStampSlots + ev] = global_ns();
  }

  // Bounded wait for ring stage `seq` to be full. False on abort / timeout.
  // Consumer warps take stages round-robin, so a warp may ask for a stage more
  // than one lap ahead of its slot; an mbarrier parity only tells adjacent
  // phases apart. The producer therefore records which stage owns a slot before
  // arming it, and the parity wait starts only once `seq` owns the slot.
  __device__ bool wait_full(long long seq) const {
    const int slot = (int)(seq % p.nslots);
    const uint32_t par = (uint32_t)((seq / p.nslots) & 1);
    const uint32_t bar = full0 + 8u * slot;
    while (slot_seq[slot] != (int)seq) {
      if (aborted()) return false;
      if (expired()) {
        fail(SITE_RING_FULL);
        return false;
      }
    }
    while (!mbar_try_wait(bar, par)) {
      if (aborted()) return false;
      if (expired()) {
        fail(SITE_RING_FULL);
        return false;
      }
    }
    return true;
  }
  // Producer side: bounded wait for the slot of stage `seq` to be free.
  __device__ bool wait_empty(long long seq) const {
    const int slot = (int)(seq % p.nslots);
    const uint32_t par = (uint32_t)(((seq / p.nslots) & 1) ^ 1);
    const uint32_t bar = empty0 + 8u * slot;
    while (!mbar_try_wait(bar, par)) {
      if (aborted()) return false;
      if (expired()) {
        fail(SITE_RING_EMPTY);
        return false;
      }
    }
    return true;
  }
  __device__ void release(long long seq, uint32_t count) const {
    mbar_arrive(empty0 + 8u * (uint32_t)(seq % p.nslots), count);
  }
};

// Routing tables in shared memory.
struct Route {
  int* sel_e;          // [maxm][K]
  float* sel_w;        // [maxm][K]
  uint32_t* emask;     // [E] row mask per expert
  int* slot_of;        // [E]
  int* slot_e;         // [nslot_max] expert id, or -1 - s for shared expert s
  uint32_t* slot_mask; // [nslot_max]
  float* slot_w;       // [nslot_max][maxm] combine weight (routed_scale folded in)
  __device__ Route(const Params& p, uint8_t* sm)
      : sel_e(reinterpret_cast<int*>(sm + p.off_sel_e)),
        sel_w(reinterpret_cast<float*>(sm + p.off_sel_w)),
        emask(reinterpret_cast<uint32_t*>(sm + p.off_emask)),
        slot_of(reinterpret_cast<int*>(sm + p.off_slot_of)),
        slot_e(reinterpret_cast<int*>(sm + p.off_slot_e)),
        slot_mask(reinterpret_cast<uint32_t*>(sm + p.off_slot_mask)),
        slot_w(reinterpret_cast<float*>(sm + p.off_slot_w)) {}
};

// --------------------------------------------------------------------------
// consumer: x rows into shared memory (optionally RMS-normalised)
// --------------------------------------------------------------------------
static __device__ void load_x(const Ctx& c) {
  const Params& p = c.p;
  uint4* xs = reinterpret_cast<uint4*>(c.sm + p.off_x);
  const int nch = p.H / 8;
  const uint4* xg = reinterpret_cast<const uint4*>(p.x);
  for (int m = c.warp; m < p.maxm; m += kNC) {
    if (m >= p.M) {
      for (int ch = c.lane; ch < nch; ch += 32) xs[m * nch + ch] = make_uint4(0, 0, 0, 0);
      continue;
    }
    float scale = 1.0f;
    if (p.pre_rmsnorm) {
      float ss = 0.0f;
      for (int ch = c.lane; ch < nch; ch += 32) {
        const uint4 v = xg[m * nch + ch];
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
      scale = 1.0f / sqrtf(ss / (float)p.H + p.rms_eps);
    }
    for (int ch = c.lane; ch < nch; ch += 32) {
      uint4 v = xg[m * nch + ch];
      if (p.pre_rmsnorm) {
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t lo = f32_to_bf16_bits(bf16lo(w[q]) * scale);
          const uint32_t hi = f32_to_bf16_bits(bf16hi(w[q]) * scale);
          w[q] = lo | (hi << 16);
        }
        v = make_uint4(w[0], w[1], w[2], w[3]);
      }
      xs[m * nch + ch] = v;
    }
  }
}

// --------------------------------------------------------------------------
// consumer: dot products of one gate/up (or router) row pair with the rows in
// `mask`. Results are warp-reduced (butterfly), so every lane holds all sums.
// --------------------------------------------------------------------------
template <int MAXM>
struct PairAcc {
  float g[MAXM];
  float u[MAXM];
};

// bf16 rows: `row_bytes` per row, stage = [row a][row b]. xr: lane's x chunks
// (MAXM == 1); xs: x rows in shared memory (MAXM > 1).
template <int MAXM, bool XREG>
__device__ __forceinline__ void pair_dot_bf16(const uint8_t* st, int row_bytes, int nch,
                                              const uint4* xr, const uint4* xs, uint32_t mask,
                                              int lane, PairAcc<MAXM>& a) {
#pragma unroll
  for (int m = 0; m < MAXM; ++m) a.g[m] = a.u[m] = 0.0f;
  const uint4* wa = reinterpret_cast<const uint4*>(st);
  const uint4* wb = reinterpret_cast<const uint4*>(st + row_bytes);
  if (MAXM == 1 && XREG) {
#pragma unroll
    for (int i = 0; i < kCplBf16; ++i) {
      const int ch = lane + 32 * i;
      if (ch < nch) {
        dot8_bf16(a.g[0], wa[ch], xr[i]);
        dot8_bf16(a.u[0], wb[ch], xr[i]);
      }
    }
  } else {
    for (int ch = lane; ch < nch; ch += 32) {
      const uint4 va = wa[ch], vb = wb[ch];
#pragma unroll
      for (int m = 0; m < MAXM; ++m) {
        if (mask >> m & 1u) {
          const uint4 xv = xs[m * nch + ch];
          dot8_bf16(a.g[m], va, xv);
          dot8_bf16(a.u[m], vb, xv);
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MAXM; ++m) {
    if (mask >> m & 1u) {
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        a.g[m] += __shfl_xor_sync(kFull, a.g[m], o);
        a.u[m] += __shfl_xor_sync(kFull, a.u[m], o);
      }
    }
  }
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

// bf16 x chunk (8 values) -> 4 fp16x2 words (exact for |x| in the fp16 range).
__device__ __forceinline__ void bf16x8_to_f16x8(const uint4 v, uint32_t* o) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half2 h = __floats2half2_rn(bf16lo(w[q]), bf16hi(w[q]));
    o[q] = *reinterpret_cast<const uint32_t*>(&h);
  }
}

// NVFP4 gate/up pair. Stage layout: [codes a][codes b][scales a][scales b].
// xr: lane's x chunks as fp16 (MAXM == 1, 16 words per chunk); xs: bf16 x rows.
template <int MAXM>
__device__ __forceinline__ void pair_dot_fp4(const uint8_t* st, int row_bytes, int sc_bytes, int nch,
                                             const uint32_t* xr, const uint4* xs, int H,
                                             uint32_t mask, int lane, PairAcc<MAXM>& a) {
#pragma unroll
  for (int m = 0; m < MAXM; ++m) a.g[m] = a.u[m] = 0.0f;
  const uint4* qa = reinterpret_cast<const uint4*>(st);
  const uint4* qb = reinterpret_cast<const uint4*>(st + row_bytes);
  const uint16_t* sa = reinterpret_cast<const uint16_t*>(st + 2 * row_bytes);
  const uint16_t* sb = reinterpret_cast<const uint16_t*>(st + 2 * row_bytes + sc_bytes);
  if (MAXM == 1) {
#pragma unroll
    for (int i = 0; i < kCplFp4; ++i) {
      const int ch = lane + 32 * i;
      if (ch < nch) {
        dot32_fp4(a.g[0], qa[ch], sa[ch], xr + 16 * i);
        dot32_fp4(a.u[0], qb[ch], sb[ch], xr + 16 * i);
      }
    }
  } else {
    for (int ch = lane; ch < nch; ch += 32) {
      const uint4 va = qa[ch], vb = qb[ch];
      const uint32_t s_a = sa[ch], s_b = sb[ch];
#pragma unroll
      for (int m = 0; m < MAXM; ++m) {
        if (mask >> m & 1u) {
          uint32_t xh[16];
          const uint4* xrow = xs + (size_t)m * (H / 8) + ch * 4;
#pragma unroll
          for (int q = 0; q < 4; ++q) bf16x8_to_f16x8(xrow[q], xh + 4 * q);
          dot32_fp4(a.g[m], va, s_a, xh);
          dot32_fp4(a.u[m], vb, s_b, xh);
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MAXM; ++m) {
    if (mask >> m & 1u) {
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        a.g[m] += __shfl_xor_sync(kFull, a.g[m], o);
        a.u[m] += __shfl_xor_sync(kFull, a.u[m], o);
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
  uint4 b[(MAXM == 1 && FMT == FMT_BF16) ? kCplBf16 : 1];         // bf16 chunks
  uint32_t h[(MAXM == 1 && FMT == FMT_NVFP4) ? 16 * kCplFp4 : 1];  // fp16 chunks (NVFP4)
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
  } else {
#pragma unroll
    for (int i = 0; i < kCplFp4; ++i) {
      const int ch = c.lane + 32 * i;  // 32-element chunk
      if (ch < p.H / 32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) bf16x8_to_f16x8(xs[ch * 4 + q], &xr.h[16 * i + 4 * q]);
      }
    }
  }
}

// Router stages: consecutive router row pairs. Writes tagged logits.
template <int FMT, int MAXM>
__device__ void consume_router(const Ctx& c, const XRegs<FMT, MAXM>& xr, long long& seq) {
  const Params& p = c.p;
  long long lo, hi;
  split_range(p.E / 2, blockIdx.x, p.grid, lo, hi);
  const long long nst = (hi - lo + p.pps_r - 1) / p.pps_r;
  const uint4* xs = reinterpret_cast<const uint4*>(c.sm + p.off_x);
  const uint32_t mask = (1u << p.M) - 1u;
  const uint32_t ep = c.epoch();
  for (long long s = c.warp; s < nst; s += kNC) {
    const long long q = seq + s;
    const bool got = !c.aborted() && c.wait_full(q);
    if (got) {
      const uint8_t* st = c.slot_ptr((int)(q % p.nslots));
      for (int it = 0; it < p.pps_r; ++it) {
        const long long item = lo + s * p.pps_r + it;
        if (item >= hi) break;
        PairAcc<MAXM> a;
        pair_dot_bf16<MAXM, FMT == FMT_BF16>(st + (size_t)it * p.rpair_bytes, p.H * 2, p.H / 8, xr.b,
                                             xs, mask, c.lane, a);
        if (!(p.test_flags & TEST_SKIP_LOGITS)) {
#pragma unroll
          for (int m = 0; m < MAXM; ++m) {
            if (c.lane == m && m < p.M) {
              st_tagged(&p.logits[(size_t)m * p.E + 2 * item], ep, a.g[m]);
              st_tagged(&p.logits[(size_t)m * p.E + 2 * item + 1], ep, a.u[m]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (got && c.lane == 0) c.release(q, kNC);
  }
  seq += nst;
}

// Gate/up stages for expert pairs. `shared_phase`: items are (shared s, j) and
// the result has weight 1; otherwise items are (routed union slot u, j).
template <int FMT, int MAXM>
__device__ void consume_pairs(const Ctx& c, const Route& rt, const XRegs<FMT, MAXM>& xr,
                              bool shared_phase, long long& seq) {
  const Params& p = c.p;
  const int n_routed = c.misc[MISC_NROUTED];
  const long long n = shared_phase ? (long long)p.S * p.I : (long long)n_routed * p.I;
  long long lo, hi;
  split_range(n, blockIdx.x, p.grid, lo, hi);
  const long long nst = (hi - lo + p.pps - 1) / p.pps;
  const uint4* xs = reinterpret_cast<const uint4*>(c.sm + p.off_x);
  const uint32_t ep = c.epoch();
  for (long long s = c.warp; s < nst; s += kNC) {
    const long long q = seq + s;
    const bool got = !c.aborted() && c.wait_full(q);
    if (got) {
      const uint8_t* st = c.slot_ptr((int)(q % p.nslots));
      for (int it = 0; it < p.pps; ++it) {
        const long long item = lo + s * p.pps + it;
        if (item >= hi) break;
        const int slot = (int)(item / p.I) + (shared_phase ? 0 : p.S);
        const int j = (int)(item % p.I);
        const uint32_t mask = shared_phase ? (1u << p.M) - 1u : rt.slot_mask[slot];
        PairAcc<MAXM> a;
        const uint8_t* pst = st + (size_t)it * p.pair_bytes;
        if (FMT == FMT_BF16)
          pair_dot_bf16<MAXM, true>(pst, p.row13, p.nchunk_h, xr.b, xs, mask, c.lane, a);
        else
          pair_dot_fp4<MAXM>(pst, p.row13, p.sc13, p.nchunk_h, xr.h, xs, p.H, mask, c.lane, a);
        float gsg = 1.0f, gsu = 1.0f;
        if (FMT == FMT_NVFP4) {
          const int e = shared_phase ? -1 - slot : rt.slot_e[slot];
          const float* gs = e >= 0 ? p.w13_gs + 2 * e : p.sh_w13_gs + 2 * (-1 - e);
          gsg = gs[0];
          gsu = gs[1];
        }
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
          if (c.lane == m && (mask >> m & 1u)) {
            const float g = a.g[m] * gsg, u = a.u[m] * gsu;
            float h = silu_f32(g) * u;
            if (!shared_phase) h *= rt.slot_w[slot * p.maxm + m];
            st_tagged(&p.hbuf[((size_t)slot * p.maxm + m) * p.I + j], ep, h);
          }
        }
      }
    }
    __syncwarp();
    if (got && c.lane == 0) c.release(q, kNC);
  }
  seq += nst;
}

// --------------------------------------------------------------------------
// consumer phase T: top-k per row and the expert union
// --------------------------------------------------------------------------
static __device__ void route_rows(const Ctx& c, const Route& rt, bool write_topk) {
  const Params& p = c.p;
  const int ctid = c.tid;  // consumers are threads [0, kNC * 32)
  const uint32_t ep = c.epoch();
  if (c.warp < p.M) {
    const int m = c.warp;
    const int P = (p.E + 31) / 32;  // logits per lane, contiguous ids
    const int base = c.lane * P;
    uint32_t key[32];
    const unsigned long long* row = p.logits + (size_t)m * p.E;
    uint64_t spins = 0;
    for (;;) {
      uint32_t bad = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        key[i] = 0;
        if (i < P && base + i < p.E) {
          unsigned long long v;
          asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(row + base + i) : "memory");
          bad |= (uint32_t)(v >> 32) != ep;
          key[i] = f32_order_key(__uint_as_float((uint32_t)v));
        }
      }
      if (!__any_sync(kFull, bad)) break;
      bool stop = c.aborted();
      if (!stop && (++spins & 63) == 0 && c.peer_failed()) stop = true;
      if (!stop && c.expired()) {
        if (c.lane == 0) c.fail(SITE_LOGITS);
        stop = true;
      }
      if (__any_sync(kFull, stop)) {
        if (c.lane == 0) *reinterpret_cast<volatile int*>(c.misc + MISC_ABORT) = 1;
#pragma unroll
        for (int i = 0; i < 32; ++i) key[i] = (i < P && base + i < p.E) ? 1u : 0u;  // any valid ids
        break;
      }
    }
    uint32_t lmax = 0;
    int lidx = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (key[i] > lmax) {
        lmax = key[i];
        lidx = i;
      }
    int my_e = 0;
    float my_v = 0.0f;
    for (int j = 0; j < p.K; ++j) {
      const uint32_t gmax = warp_max_u32(lmax);
      const int winner = __ffs(__ballot_sync(kFull, lmax == gmax)) - 1;
      const int e = __shfl_sync(kFull, base + lidx, winner);
      if (c.lane == j) {
        my_e = e;
        my_v = order_key_f32(gmax);
      }
      if (c.lane == winner) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i == lidx) key[i] = 0;
        lmax = 0;
        lidx = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (key[i] > lmax) {
            lmax = key[i];
            lidx = i;
          }
      }
    }
    const float v0 = __shfl_sync(kFull, my_v, 0);
    float ex = c.lane < p.K ? expf(my_v - v0) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
    if (c.lane < p.K) {
      const float w = ex / sum;
      rt.sel_e[m * p.K + c.lane] = my_e;
      rt.sel_w[m * p.K + c.lane] = w;
      if (write_topk && blockIdx.x == 0) {
        if (p.topk_idx) p.topk_idx[m * p.K + c.lane] = my_e;
        if (p.topk_w) p.topk_w[m * p.K + c.lane] = w;
      }
    }
  }
  bar_sync(kBarConsumers, kNC * 32);
  for (int t = ctid; t < p.M * p.K; t += kNC * 32) atomicOr(&rt.emask[rt.sel_e[t]], 1u << (t / p.K));
  bar_sync(kBarConsumers, kNC * 32);
  // Compact the experts with a non-zero row mask, ascending id (popcount prefix).
  int* wtot = c.misc + MISC_WTOT;
  int running = 0;
  for (int e0 = 0; e0 < p.E; e0 += kNC * 32) {
    const int e = e0 + ctid;
    const bool nz = e < p.E && rt.emask[e] != 0u;
    const uint32_t bal = __ballot_sync(kFull, nz);
    if (c.lane == 0) wtot[c.warp] = __popc(bal);
    bar_sync(kBarConsumers, kNC * 32);
    int before = 0, total = 0;
    for (int w = 0; w < kNC; ++w) {
      const int v = wtot[w];
      before += w < c.warp ? v : 0;
      total += v;
    }
    if (nz) {
      const int s = p.S + running + before + __popc(bal & lanemask_lt());
      rt.slot_of[e] = s;
      rt.slot_e[s] = e;
      rt.slot_mask[s] = rt.emask[e];
    }
    running += total;
    bar_sync(kBarConsumers, kNC * 32);
  }
  if (ctid == 0) c.misc[MISC_NROUTED] = running;
  for (int t = ctid; t < p.S; t += kNC * 32) {
    rt.slot_e[t] = -1 - t;
    rt.slot_mask[t] = (1u << p.M) - 1u;
    for (int m = 0; m < p.maxm; ++m) rt.slot_w[t * p.maxm + m] = 1.0f;
  }
  for (int t = ctid; t < p.M * p.K; t += kNC * 32)
    rt.slot_w[rt.slot_of[rt.sel_e[t]] * p.maxm + t / p.K] = rt.sel_w[t] * p.routed_scale;
  bar_sync(kBarConsumers, kNC * 32);
}

// --------------------------------------------------------------------------
// consumer phase D
// --------------------------------------------------------------------------
__device__ __forceinline__ void cta_rows(const Params& p, int& r_lo, int& r_hi) {
  long long lo, hi;
  split_range(p.H, blockIdx.x, p.grid, lo, hi);
  r_lo = (int)lo;
  r_hi = (int)hi;
}

// Wait until every CTA has copied x into shared memory (only needed when the
// output overwrites x in the single-kernel schedule).
static __device__ bool wait_xflags(const Ctx& c) {
  const Params& p = c.p;
  const uint32_t ep = c.epoch();
  uint64_t spins = 0;
  for (int i = c.tid; i < p.grid; i += kNC * 32) {
    for (;;) {
      unsigned long long v;
      asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p.xflags + i) : "memory");
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

// check_xflags: the output overwrites x and other CTAs of this kernel may still
// be reading x (single-kernel schedule only).
template <int FMT, int MAXM>
__device__ void consume_down(const Ctx& c, const Route& rt, bool check_xflags, long long& seq) {
  const Params& p = c.p;
  int r_lo, r_hi;
  cta_rows(p, r_lo, r_hi);
  const int drs = p.d_rows_stage;
  const int nrb = (r_hi - r_lo + drs - 1) / drs;
  const int nsl = p.S + c.misc[MISC_NROUTED];
  const int ctid = c.tid;
  const int g = ctid / p.tg;        // thread group
  const int ch = ctid % p.tg;       // 16-byte code chunk of a down row
  const bool active = g < p.ng;
  const uint32_t ep = c.epoch();
  float* hs0 = reinterpret_cast<float*>(c.sm + p.off_hs);
  float* red = reinterpret_cast<float*>(c.sm + p.off_red);
  const int hs_words = p.maxm * p.I;
  constexpr int CH_EL = FMT == FMT_BF16 ? 8 : 32;  // elements per chunk
  int buf = 0;
  for (int rb = 0; rb < nrb; ++rb) {
    const int rb_lo = r_lo + rb * drs;
    const int nr = min(drs, r_hi - rb_lo);
    float acc[kRpgMax][MAXM];
#pragma unroll
    for (int ri = 0; ri < kRpgMax; ++ri)
#pragma unroll
      for (int m = 0; m < MAXM; ++m) acc[ri][m] = 0.0f;
    for (int sl = 0; sl < nsl; ++sl, ++seq) {
      const uint32_t mask = rt.slot_mask[sl];
      float* hs = hs0 + buf * hs_words;
      // Stage this expert's h rows (tagged, from every CTA) into shared memory.
      bool ok = !c.aborted();
      if (ok) {
        uint64_t spins = 0;
        const int pairs = p.M * p.I / 2;
        for (int t = ctid; t < pairs && ok; t += kNC * 32) {
          const int m = (2 * t) / p.I;
          if (!(mask >> m & 1u)) continue;
          const int k = (2 * t) % p.I;
          const unsigned long long* src = p.hbuf + ((size_t)sl * p.maxm + m) * p.I + k;
          for (;;) {
            unsigned long long v0, v1;
            ld_tagged2(src, v0, v1);
            if ((uint32_t)(v0 >> 32) == ep && (uint32_t)(v1 >> 32) == ep) {
              hs[m * p.I + k] = __uint_as_float((uint32_t)v0);
              hs[m * p.I + k + 1] = __uint_as_float((uint32_t)v1);
              break;
            }
            if (c.aborted() || ((++spins & 63) == 0 && c.peer_failed())) {
              ok = false;
              break;
            }
            if (c.expired()) {
              c.fail(SITE_HIDDEN);
              ok = false;
              break;
            }
          }
        }
      }
      const bool got = ok && !c.aborted() && c.wait_full(seq);
      ok = got;
      bar_sync(kBarConsumers, kNC * 32);
      if (rb == 0 && sl == 0 && c.tid == 0) c.stamp(ST_D_FIRST);
      if (ok && !c.aborted() && active) {
        const uint8_t* st = c.slot_ptr((int)(seq % p.nslots));
        float gsc = 1.0f;
        if (FMT == FMT_NVFP4) {
          const int e = rt.slot_e[sl];
          gsc = e >= 0 ? p.w2_gs[e] : p.sh_w2_gs[-1 - e];
        }
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
          if (!(mask >> m & 1u)) continue;
          float hv[CH_EL];
          const float4* hp = reinterpret_cast<const float4*>(hs + m * p.I + ch * CH_EL);
#pragma unroll
          for (int q = 0; q < CH_EL / 4; ++q) {
            const float4 f = hp[q];
            hv[4 * q] = f.x * gsc;
            hv[4 * q + 1] = f.y * gsc;
            hv[4 * q + 2] = f.z * gsc;
            hv[4 * q + 3] = f.w * gsc;
          }
#pragma unroll
          for (int ri = 0; ri < kRpgMax; ++ri) {
            const int r = g + ri * p.ng;
            if (r < nr) {
              if (FMT == FMT_BF16) {
                const uint4 w = reinterpret_cast<const uint4*>(st + (size_t)r * p.row2)[ch];
                dot8_bf16_f32(acc[ri][m], w, hv);
              } else {
                const uint4 qv = reinterpret_cast<const uint4*>(st + (size_t)r * p.row2)[ch];
                const uint32_t sc = reinterpret_cast<const uint16_t*>(
                    st + (size_t)drs * p.row2 + (size_t)r * p.sc2)[ch];
                const uint32_t sf = e4m3x2_to_f16x2(sc);
                const float s[2] = {__half2float(__ushort_as_half((unsigned short)(sf & 0xffffu))),
                                    __half2float(__ushort_as_half((unsigned short)(sf >> 16)))};
                const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                  float part = 0.0f;
#pragma unroll
                  for (int wi = 0; wi < 2; ++wi) {
#pragma unroll
                    for (int by = 0; by < 4; ++by) {
                      const uint32_t wv = e2m1x2_to_f16x2((qw[blk * 2 + wi] >> (8 * by)) & 0xffu);
                      const int e0 = blk * 16 + wi * 8 + by * 2;
                      const __half2 wh = *reinterpret_cast<const __half2*>(&wv);
                      part = fmaf(__low2float(wh), hv[e0], part);
                      part = fmaf(__high2float(wh), hv[e0 + 1], part);
                    }
                  }
                  acc[ri][m] = fmaf(s[blk], part, acc[ri][m]);
                }
              }
            }
          }
        }
      }
      __syncwarp();
      if (got && c.lane == 0) c.release(seq, 1);
      buf ^= 1;
    }
    // Reduce each row's partial sums over the group's threads and write out.
    if (check_xflags && rb == 0) {
      if (!c.aborted()) wait_xflags(c);
      bar_sync(kBarConsumers, kNC * 32);
    }
    const bool write = !c.aborted();
    if (p.tg <= 32) {
#pragma unroll
      for (int ri = 0; ri < kRpgMax; ++ri)
#pragma unroll
        for (int m = 0; m < MAXM; ++m)
          for (int o = p.tg >> 1; o; o >>= 1) acc[ri][m] += __shfl_xor_sync(kFull, acc[ri][m], o);
      if (write && active && ch == 0) {
#pragma unroll
        for (int ri = 0; ri < kRpgMax; ++ri) {
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
      for (int ri = 0; ri < kRpgMax; ++ri)
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
          float v = acc[ri][m];
#pragma unroll
          for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
          if (c.lane == 0) red[(c.warp * kRpgMax + ri) * MAXM + m] = v;
        }
      bar_sync(kBarConsumers, kNC * 32);
      const int wpg = p.tg / 32;
      if (write && active && ch < 32) {  // first warp of each group writes
        for (int q = c.lane; q < kRpgMax * MAXM; q += 32) {
          const int ri = q / MAXM, m = q % MAXM;
          const int r = g + ri * p.ng;
          if (r < nr && m < p.M) {
            float y = 0.0f;
            for (int w = 0; w < wpg; ++w) y += red[((g * wpg + w) * kRpgMax + ri) * MAXM + m];
            const int row = rb_lo + r;
            const float rv = __uint_as_float((uint32_t)p.resid[(size_t)m * p.H + row] << 16);
            p.out[(size_t)m * p.H + row] = f32_to_bf16_bits(rv + y);
          }
        }
      }
      bar_sync(kBarConsumers, kNC * 32);
    }
  }
}

// --------------------------------------------------------------------------
// producer (lane 0 of the last warp issues; the warp stays converged)
// --------------------------------------------------------------------------
struct Producer {
  const Ctx& c;
  uint64_t pol;
  long long issued = 0;  // stages whose copies were issued
  __device__ Producer(const Ctx& cc) : c(cc) { pol = policy_evict_first(); }

  // Claims the next stage's slot and announces its bytes. False on abort.
  __device__ bool begin(long long seq, uint32_t bytes, uint32_t& dst, uint32_t& bar) {
    if (c.aborted() || !c.wait_empty(seq)) return false;
    const int slot = (int)(seq % c.p.nslots);
    dst = smem_u32(c.slot_ptr(slot));
    bar = c.full0 + 8u * slot;
    c.slot_seq[slot] = (int)seq;  // before arming: see Ctx::wait_full
    mbar_arrive_expect_tx(bar, bytes);
    issued = seq + 1;
    return true;
  }

  __device__ void router(long long& seq) {
    const Params& p = c.p;
    long long lo, hi;
    split_range(p.E / 2, blockIdx.x, p.grid, lo, hi);
    const long long nst = (hi - lo + p.pps_r - 1) / p.pps_r;
    for (long long s = 0; s < nst; ++s) {
      const long long a = lo + s * p.pps_r, b = min(hi, a + p.pps_r);
      const uint32_t bytes = (uint32_t)((b - a) * p.rpair_bytes);
      uint32_t dst, bar;
      if (!begin(seq + s, bytes, dst, bar)) break;
      bulk_g2s(dst, p.router_w + (size_t)a * p.rpair_bytes, bytes, bar, pol);
    }
    seq += nst;
  }

  // Gate/up row pairs: shared experts (shared_phase) or the routed union.
  __device__ void pairs(bool shared_phase, const Route& rt, long long& seq) {
    const Params& p = c.p;
    const int n_routed = c.misc[MISC_NROUTED];
    const long long n = shared_phase ? (long long)p.S * p.I : (long long)n_routed * p.I;
    long long lo, hi;
    split_range(n, blockIdx.x, p.grid, lo, hi);
    const long long nst = (hi - lo + p.pps - 1) / p.pps;
    for (long long s = 0; s < nst; ++s) {
      const long long a = lo + s * p.pps, b = min(hi, a + p.pps);
      uint32_t dst, bar;
      if (!begin(seq + s, (uint32_t)((b - a) * p.pair_bytes), dst, bar)) break;
      for (long long item = a; item < b; ++item) {
        const int slot = (int)(item / p.I) + (shared_phase ? 0 : p.S);
        const int j = (int)(item % p.I);
        const int e = shared_phase ? -1 - slot : rt.slot_e[slot];
        const uint8_t* w = e >= 0 ? p.w13 : p.sh_w13;
        const uint8_t* ws = e >= 0 ? p.w13_s : p.sh_w13_s;
        const size_t ex = (size_t)(e >= 0 ? e : -1 - e);
        const size_t rg = ex * 2 * p.I + j, ru = rg + p.I;  // gate row, up row
        const uint32_t d = dst + (uint32_t)((item - a) * p.pair_bytes);
        bulk_g2s(d, w + rg * p.row13, p.row13, bar, pol);
        bulk_g2s(d + p.row13, w + ru * p.row13, p.row13, bar, pol);
        if (p.sc13) {
          bulk_g2s(d + 2 * p.row13, ws + rg * p.sc13, p.sc13, bar, pol);
          bulk_g2s(d + 2 * p.row13 + p.sc13, ws + ru * p.sc13, p.sc13, bar, pol);
        }
      }
    }
    seq += nst;
  }

  // Down stages (row block rb, union slot sl) for sl in [sl_lo, sl_hi) of block rb.
  __device__ void down_block(const Route& rt, int rb, int sl_lo, int sl_hi, long long& seq) {
    const Params& p = c.p;
    int r_lo, r_hi;
    cta_rows(p, r_lo, r_hi);
    const int rb_lo = r_lo + rb * p.d_rows_stage;
    const int nr = min(p.d_rows_stage, r_hi - rb_lo);
    for (int sl = sl_lo; sl < sl_hi; ++sl, ++seq) {
      const int e = sl < p.S ? -1 - sl : rt.slot_e[sl];
      const uint8_t* w = e >= 0 ? p.w2 : p.sh_w2;
      const uint8_t* ws = e >= 0 ? p.w2_s : p.sh_w2_s;
      const size_t ex = (size_t)(e >= 0 ? e : -1 - e);
      const size_t row0 = ex * p.H + rb_lo;
      const uint32_t cb = (uint32_t)nr * p.row2, sb = (uint32_t)nr * p.sc2;
      uint32_t dst, bar;
      if (!begin(seq, cb + sb, dst, bar)) {
        seq = seq + (sl_hi - sl);
        return;
      }
      bulk_g2s(dst, w + row0 * p.row2, cb, bar, pol);
      if (sb) bulk_g2s(dst + (uint32_t)p.d_rows_stage * p.row2, ws + row0 * p.sc2, sb, bar, pol);
    }
  }

  __device__ int down_blocks() const {
    int r_lo, r_hi;
    cta_rows(c.p, r_lo, r_hi);
    return (r_hi - r_lo + c.p.d_rows_stage - 1) / c.p.d_rows_stage;
  }

  // Shared experts' down rows of this CTA into L2 ahead of time.
  __device__ void prefetch_shared_down() {
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

  // After an abort: wait (bounded) for this CTA's copies still in flight.
  __device__ void drain() {
    const Params& p = c.p;
    const long long first = issued > p.nslots ? issued - p.nslots : 0;
    const uint64_t t = global_ns();
    for (long long q = first; q < issued; ++q) {
      const uint32_t bar = c.full0 + 8u * (uint32_t)(q % p.nslots);
      const uint32_t par = (uint32_t)((q / p.nslots) & 1);
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
    for (int i = 0; i < p.nslots; ++i) {
      mbar_init(c.full0 + 8u * i, 1);
      mbar_init(c.empty0 + 8u * i, kNC);
      c.slot_seq[i] = -1;
    }
    mbar_init_fence();
    c.misc[MISC_ABORT] = 0;
    c.misc[MISC_NROUTED] = 0;
  }
  for (int e = c.tid; e < p.E; e += kThreads) rt.emask[e] = 0u;
  __syncthreads();

  if (c.warp == kNC) {
    // ------------------------------------------------------------ producer
    Producer pr(c);
    long long seq = 0;
    if (PHASES & PH_R) {
      if (c.lane == 0) {
        pr.router(seq);
        pr.pairs(true, rt, seq);
        c.stamp(ST_P_R_ISSUED);
        if (PHASES & PH_D) pr.prefetch_shared_down();
      }
    } else if (PHASES == PH_D) {
      // The shared experts' down rows of the first row block need no routing.
      if (c.lane == 0 && pr.down_blocks() > 0) pr.down_block(rt, 0, 0, p.S, seq);
    }
    if (kRoute) {
      __syncwarp();
      bar_sync(kBarRoute, kThreads);
    }
    if (c.lane == 0) {
      c.stamp(ST_P_ROUTE);
      if (PHASES & PH_U) {
        pr.pairs(false, rt, seq);
        c.stamp(ST_P_U_ISSUED);
      }
      if (PHASES & PH_D) {
        const int nsl = p.S + c.misc[MISC_NROUTED];
        const int first = PHASES == PH_D ? p.S : 0;  // the chain issued these before routing
        for (int rb = 0; rb < pr.down_blocks(); ++rb) pr.down_block(rt, rb, rb == 0 ? first : 0, nsl, seq);
        c.stamp(ST_P_D_ISSUED);
      }
      if (c.aborted()) pr.drain();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    if (kChain) pdl_wait();
    if (c.tid == 0) c.misc[MISC_EPOCH] = (int)ld_relaxed_u32(&p.ctrl[CTRL_EPOCH]);
    if (c.tid == 0) c.stamp(ST_START);
    if (kNeedX) load_x(c);
    bar_sync(kBarConsumers, kNC * 32);
    if (c.tid == 0) c.stamp(ST_X_LOADED);
    if (PHASES == PH_ALL && p.out_aliases_x && c.tid == 0)
      st_tagged(p.xflags + blockIdx.x, c.epoch(), 0.0f);
    long long seq = 0;
    if (PHASES & PH_R) {
      XRegs<FMT, MAXM> xr;
      load_xregs<FMT, MAXM>(c, xr);
      consume_router<FMT, MAXM>(c, xr, seq);
      consume_pairs<FMT, MAXM>(c, rt, xr, true, seq);
      if (c.tid == 0) c.stamp(ST_R_DONE);
    }
    if (kRoute) {
      route_rows(c, rt, (PHASES & PH_U) != 0);
      bar_arrive(kBarRoute, kThreads);
      if (c.tid == 0) c.stamp(ST_ROUTED);
    }
    if (PHASES & PH_U) {
      XRegs<FMT, MAXM> xr;
      load_xregs<FMT, MAXM>(c, xr);
      consume_pairs<FMT, MAXM>(c, rt, xr, false, seq);
      if (c.tid == 0) c.stamp(ST_U_DONE);
    }
    if (PHASES & PH_D) consume_down<FMT, MAXM>(c, rt, PHASES == PH_ALL && p.out_aliases_x, seq);
    if (c.tid == 0) c.stamp(ST_D_DONE);
  }
  __syncthreads();
  if (kLast && c.tid == 0) {
    const uint32_t prev = atomicAdd(&p.ctrl[CTRL_EXIT], 1u);
    if (prev == gridDim.x - 1) {
      p.ctrl[CTRL_EXIT] = 0u;
      uint32_t e = p.ctrl[CTRL_EPOCH] + 1u;
      if (e == 0xffffffffu) e = 0u;
      p.ctrl[CTRL_EPOCH] = e;
    }
  }
}

}  // namespace moe
