// The split-K single kernel: the expert down matrices are stored transposed
// ([I][H] per expert, so the down weights of one h row are one contiguous row).
// Each CTA owns a contiguous range of (expert, intermediate row) items -- the
// shared experts' rows, then the routed experts' rows of the union -- and for
// every item streams the gate row, the up row and the transposed down row. It
// computes the item's h values (SiLU(gate) * up, times the routing weight) into
// shared memory and adds their down-projection contributions to per-thread
// partial sums over all H outputs. No h row crosses CTAs: the only exchange is
// the final one, where every CTA stores its partial sums, and each CTA reduces
// its block of output rows over all CTAs' partials in a fixed order (the same
// result every run), adds the residual and rounds once to bf16.
//
// "Muse Spark Open Ultrafast", section "A new tensor parallelism", names the two
// ways to split the expert GEMMs over workers: the second GEMM split on the
// intermediate dimension with one reduction at the end, or both split on the
// output dimension with the intermediate values gathered in between. The
// row-block schedules of this library do the latter across the CTAs of one GPU;
// this kernel does the former. The layer it computes is the same (the Ling
// blog's MoE chain of "PDL: stacking the latency floors of small kernels": up
// GEMM, activation, down GEMM, combine as an fp32 sum with one final cast); only
// the order in which the down projection's products are summed differs.
#pragma once

#include "moe_kernels.cuh"

namespace moe {

// The stage order of one range of items [lo, hi): gate/up stages of q rows and
// transposed-down stages of dq rows, neither crossing an expert; a down stage
// is taken once the gate/up stages have passed its last row by `lag` rows (or
// at the end of the range), so its h rows are normally stored by then.
struct SkSeq {
  ItemWalk gu, dn;
  int lag;
  __device__ __forceinline__ SkSeq(int lo, int hi, int q, int dq, int I, int lag_)
      : gu(lo, hi, q, I), dn(lo, hi, dq, I), lag(lag_) {}
  // 0: done, 1: the next stage is gate/up (gu), 2: it is a down stage (dn)
  __device__ __forceinline__ int kind() const {
    if (dn.more() && (!gu.more() || dn.a + dn.count() + lag <= gu.a)) return 2;
    return gu.more() ? 1 : 0;
  }
};

// The CTA whose output block (split_range of H over the grid) holds row r.
__device__ __forceinline__ int sk_owner(int r, int H, int grid) { return ((r + 1) * grid + H - 1) / H - 1; }

template <int FMT>
__device__ __forceinline__ uint32_t sk_w2t_row_bytes(const Params& p) {
  return (uint32_t)p.H * (FMT == FMT_BF16 ? 2u : 1u);
}

// Transposed down rows i0 .. i0 + nd - 1 of expert e (shared expert -1 - e).
template <int FMT>
__device__ __forceinline__ void sk_copy_w2t(const Producer& pr, int e, int i0, int nd, uint32_t dst, uint32_t bar) {
  const Params& p = pr.c.p;
  const uint8_t* wt = e >= 0 ? p.w2 : p.sh_w2;
  const size_t ex = (size_t)(e >= 0 ? e : -1 - e);
  const uint32_t rb = sk_w2t_row_bytes<FMT>(p);
  bulk_g2s(dst, wt + (ex * p.I + i0) * rb, (uint32_t)nd * rb, bar, pr.pol);
}

// Producer: the stages of one range, in the order of SkSeq.
template <int FMT>
__device__ __forceinline__ void sk_produce(Producer& pr, const Route& rt, int lo, int hi, bool shared) {
  const Params& p = pr.c.p;
  const uint32_t rb = sk_w2t_row_bytes<FMT>(p);
  for (SkSeq q(lo, hi, p.q, p.dq, p.I, p.sk_lag);; pr.ring.next(p.nslots)) {
    const int k = q.kind();
    if (k == 0) break;
    uint32_t dst, bar;
    if (k == 1) {
      const int nq = q.gu.count();
      const int slot = q.gu.u + (shared ? 0 : p.S);
      if (!pr.begin((uint32_t)nq * p.pair_bytes, dst, bar)) return;
      pr.copy_pairs(shared ? -1 - slot : rt.slot_e[slot], q.gu.j, nq, dst, bar);
      q.gu.advance(nq);
    } else {
      const int nd = q.dn.count();
      const int slot = q.dn.u + (shared ? 0 : p.S);
      if (!pr.begin((uint32_t)nd * rb, dst, bar)) return;
      sk_copy_w2t<FMT>(pr, shared ? -1 - slot : rt.slot_e[slot], q.dn.j, nd, dst, bar);
      q.dn.advance(nd);
    }
  }
}

// Bounded wait until the tag of h row r is set (every consumer thread polls the
// same shared-memory word).
__device__ __forceinline__ bool sk_wait_row(const Ctx& c, const volatile int* tag) {
  for (uint32_t spin = 0; *tag == 0; ++spin) {
    __nanosleep(32);
    if ((spin & 15) == 15) {
      if (c.aborted()) return false;
      if (c.expired()) {
        c.fail(SITE_HIDDEN);
        return false;
      }
    }
  }
  __threadfence_block();  // the row's h values after its tag
  return true;
}

// One down stage (every consumer warp): transposed down rows i0 .. i0 + nd - 1
// of the slot's expert against the stored h of those rows; thread t adds to the
// partial sums of outputs 8t .. 8t + 7 (t < H / 8), for each row of x that chose
// the expert. FP8: e4m3 codes times the block scale of (row, output column).
template <int FMT, int MAXM>
__device__ __forceinline__ Ring sk_down(const Ctx& c, const Route& rt, Ring ring, int slot, bool shared, int i0,
                                        int nd, const float* hsk, const volatile int* htag,
                                        float (&acc)[8][MAXM]) {
  const Params& p = c.p;
  const int t = c.tid;
  const bool active = t < p.H / 8;
  const uint32_t mask = shared ? (1u << p.M) - 1u : rt.slot_mask[slot];
  bool ok = !c.aborted() && c.wait_full(ring);
  for (int rr = 0; ok && rr < nd; ++rr) ok = sk_wait_row(c, htag + rr);
  if (ok && active) {
    const uint8_t* st = c.slot_ptr(ring.slot);
    const uint32_t rb = sk_w2t_row_bytes<FMT>(p);
    const float* s2 = nullptr;
    if (FMT == FMT_FP8) {
      const int e = shared ? -1 - slot : rt.slot_e[slot];
      s2 = reinterpret_cast<const float*>(e >= 0 ? p.w2_s : p.sh_w2_s) +
           (size_t)(e >= 0 ? e : -1 - e) * (p.I / kFp8Block) * (p.H / kFp8Block) + (8 * t) / kFp8Block;
    }
#pragma unroll 2
    for (int rr = 0; rr < nd; ++rr) {
      float w[8];
      if (FMT == FMT_BF16) {
        const uint4 v = reinterpret_cast<const uint4*>(st + (size_t)rr * rb)[t];
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          w[2 * k] = bf16lo(w4[k]);
          w[2 * k + 1] = bf16hi(w4[k]);
        }
      } else {
        const uint2 v = reinterpret_cast<const uint2*>(st + (size_t)rr * rb)[t];
        const float sc = __ldg(s2 + (size_t)((i0 + rr) / kFp8Block) * (p.H / kFp8Block));
        const uint32_t q2[2] = {v.x, v.y};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t f = e4m3x2_to_f16x2((q2[k >> 1] >> (16 * (k & 1))) & 0xffffu);
          const __half2 h2 = *reinterpret_cast<const __half2*>(&f);
          w[2 * k] = __low2float(h2) * sc;
          w[2 * k + 1] = __high2float(h2) * sc;
        }
      }
      const float* hr = hsk + (size_t)rr * p.maxm;
#pragma unroll
      for (int m = 0; m < MAXM; ++m) {
        if (!(mask >> m & 1u)) continue;
        const float hv = hr[m];
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k][m] = fmaf(w[k], hv, acc[k][m]);
      }
    }
  }
  __syncwarp();
  if (c.lane == 0 && ok) c.release(ring, 1);
  ring.next(p.nslots);
  return ring;
}

// Consumers: the stages of one range. rbase: this CTA's h row of the range's first item.
template <int FMT, int MAXM>
__device__ __forceinline__ Ring sk_consume(const Ctx& c, const Route& rt, Ring ring, int lo, int hi, bool shared,
                                           int rbase, const XRegs<FMT, MAXM>& xr, float (&acc)[8][MAXM]) {
  const Params& p = c.p;
  const uint4* xs = reinterpret_cast<const uint4*>(c.sm + p.off_x);
  float* hsk = reinterpret_cast<float*>(c.sm + p.off_hsk);
  volatile int* htag = reinterpret_cast<volatile int*>(c.sm + p.off_htag);
  const int slot0 = shared ? 0 : p.S;
  for (SkSeq q(lo, hi, p.q, p.dq, p.I, p.sk_lag);;) {
    const int k = q.kind();
    if (k == 0) break;
    if (k == 1) {
      const int r0 = rbase + (q.gu.a - lo);
      // the host plans sk_rows_max from the largest split; past it this CTA
      // stops (no store out of the h area)
      if (r0 + q.gu.count() > p.sk_rows_max && !c.aborted()) c.fail(SITE_FLAGS);
      item_stage<FMT, MAXM>(c, rt, q.gu, ring, slot0 + q.gu.u, shared, xr, xs, false, hsk + (size_t)r0 * p.maxm,
                            htag + r0);
      q.gu.advance(q.gu.count());
      ring.next(p.nslots);
    } else {
      const int r0 = rbase + (q.dn.a - lo);
      ring = sk_down<FMT, MAXM>(c, rt, ring, slot0 + q.dn.u, shared, q.dn.j, q.dn.count(),
                                hsk + (size_t)r0 * p.maxm, htag + r0, acc);
      q.dn.advance(q.dn.count());
    }
  }
  return ring;
}

// The final exchange: every CTA's partial sums into the destination blocks'
// areas, one count, then each CTA's block (all sources, in source order) into
// shared memory by one bulk copy, a fixed-order sum, the residual and one bf16
// rounding.
template <int FMT, int MAXM>
__device__ __forceinline__ void sk_finish(const Ctx& c, float (&acc)[8][MAXM]) {
  const Params& p = c.p;
  const int t = c.tid, M = p.M, G = p.grid;
  if (t < p.H / 8) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int row = 8 * t + k;
      const int b = sk_owner(row, p.H, G);
      int blo, bhi;
      split_range(p.H, b, G, blo, bhi);
      float* dst = p.psum + (((size_t)b * G + blockIdx.x) * M) * p.nrp + (row - blo);
#pragma unroll
      for (int m = 0; m < MAXM; ++m)
        if (m < M) __stcg(dst + (size_t)m * p.nrp, acc[k][m]);
    }
  }
  bar_sync(kBarConsumers, kNC * 32);
  const uint32_t psb = smem_u32(c.sm + p.off_psb);
  const uint32_t bytes = (uint32_t)G * M * p.nrp * 4u;
  float* stage = reinterpret_cast<float*>(c.sm + p.off_ring);
  bool issued = false;  // thread 0: the block's copy is in flight
  if (t == 0) {
    __threadfence();  // this CTA's partial sums before its count
    count_done(p, CTRL_UCOUNT);
    if (!c.aborted() && wait_count(c, CTRL_UCOUNT, SITE_FLAGS)) {
      issued = true;
      c.stamp(ST_U_FLAGS);
      __threadfence();
      fence_proxy_async_global();  // the acquired partial sums before the bulk copy that reads them
      mbar_arrive_expect_tx(psb, bytes);
      bulk_g2s_plain(smem_u32(stage), p.psum + (size_t)blockIdx.x * G * M * p.nrp, bytes, psb);
    } else {
      c.abort_local();
    }
  }
  bar_sync(kBarConsumers, kNC * 32);
  if (c.aborted()) {
    // a copy issued before the abort lands (bounded) before exit
    if (issued) {
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(psb, 0) && global_ns() - t0 < p.timeout_ns) {
      }
    }
    return;
  }
  if (!c.wait_bar(psb, 0, SITE_HIDDEN)) return;
  int r_lo, r_hi;
  split_range(p.H, blockIdx.x, G, r_lo, r_hi);
  const int nr = r_hi - r_lo;
  const int pairs = M * nr;
  if (pairs == 0) return;
  const int parts = max(1, min(G, kNC * 32 / pairs));
  float* red = reinterpret_cast<float*>(c.sm + p.off_psum);
  if (t < pairs * parts) {
    const int pr = t / parts, part = t - pr * parts;
    const int m = pr / nr, rr = pr - m * nr;
    int c0, c1;
    split_range(G, part, parts, c0, c1);
    float s = 0.0f;
    for (int src = c0; src < c1; ++src) s += stage[((size_t)src * M + m) * p.nrp + rr];
    red[t] = s;
  }
  bar_sync(kBarConsumers, kNC * 32);
  if (t < pairs && !c.aborted()) {
    const int m = t / nr, rr = t - m * nr;
    float s = 0.0f;
    for (int part = 0; part < parts; ++part) s += red[t * parts + part];
    const size_t at = (size_t)m * p.H + r_lo + rr;
    const float r = __uint_as_float((uint32_t)p.resid[at] << 16);
    p.out[at] = f32_to_bf16_bits(r + s);
  }
}

template <int FMT, int MAXM>
__global__ void __launch_bounds__(kThreads, 1) moe_sk_kernel(const __grid_constant__ Params p) {
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
    mbar_init(smem_u32(sm + p.off_psb), 1);
    mbar_init_fence();
    c.misc[MISC_ABORT] = 0;
    c.misc[MISC_NROUTED] = 0;
    c.misc[MISC_ROUTED] = 0;
  }
  for (int e = c.tid; e < p.E; e += kThreads) rt.emask[e] = 0u;
  for (int e = c.tid; e < (p.E + 31) / 32; e += kThreads) rt.bitmap[e] = 0u;
  for (int r = c.tid; r < p.sk_rows_max; r += kThreads) reinterpret_cast<int*>(sm + p.off_htag)[r] = 0;
  __syncthreads();

  int s_lo, s_hi;  // this CTA's shared-expert items
  split_range(p.S * p.I, blockIdx.x, p.grid, s_lo, s_hi);
  if (c.warp == kNC) {
    // ------------------------------------------------------------ producer
    Producer pr(c);
    if (c.lane == 0) {
      c.stamp(ST_START);
      pr.x_rows();
      pr.router();
      sk_produce<FMT>(pr, rt, s_lo, s_hi, true);
      c.stamp(ST_P_R_ISSUED);
      pr.prefetch_predicted();
    }
    __syncwarp();
    bar_sync(kBarRoute, kThreads);
    if (c.lane == 0) {
      c.stamp(ST_P_ROUTE);
      sk_produce<FMT>(pr, rt, c.misc[MISC_ULO], c.misc[MISC_UHI], false);
      c.stamp(ST_P_U_ISSUED);
      if (c.aborted()) {
        pr.drain();
        const uint64_t t = global_ns();
        while (!mbar_try_wait(c.xbar, 0) && global_ns() - t < p.timeout_ns) {
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    if (c.tid == 0) c.misc[MISC_EPOCH] = (int)ld_relaxed_u32(&p.ctrl[CTRL_EPOCH]);
    prepare_x(c, FMT != FMT_BF16);
    bar_sync(kBarConsumers, kNC * 32);
    if (c.tid == 0) c.stamp(ST_X_LOADED);
    Ring ring;
    ring = consume_router<MAXM>(c, ring);
    bar_sync(kBarConsumers, kNC * 32);  // this CTA's logits are all stored
    if (c.tid == 0) {
      c.stamp(ST_RFLAG);
    }
    route_rows<MAXM>(c, rt, true);
    if (c.tid == 0) reinterpret_cast<volatile int*>(c.misc)[MISC_ROUTED] = 1;  // hint for the producer's prefetch
    bar_arrive(kBarRoute, kThreads);
    if (c.tid == 0) c.stamp(ST_ROUTED);
    if (FMT != FMT_BF16) {  // the router is done with the bf16 x rows
      x_to_f16(c);
      bar_sync(kBarConsumers, kNC * 32);
    }
    XRegs<FMT, MAXM> xr;
    load_xregs<FMT, MAXM>(c, xr);
    float acc[8][MAXM];
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
      for (int m = 0; m < MAXM; ++m) acc[k][m] = 0.0f;
    ring = sk_consume<FMT, MAXM>(c, rt, ring, s_lo, s_hi, true, 0, xr, acc);
    if (c.tid == 0) c.stamp(ST_R_DONE);
    ring = sk_consume<FMT, MAXM>(c, rt, ring, c.misc[MISC_ULO], c.misc[MISC_UHI], false, s_hi - s_lo, xr, acc);
    if (c.tid == 0) c.stamp(ST_U_DONE);
    sk_finish<FMT, MAXM>(c, acc);
    write_prediction(c, rt);
    if (c.tid == 0) {
      c.stamp(ST_D_DONE);
      if (p.stamps) {
        p.stamps[(size_t)blockIdx.x * kStampSlots + ST_CLOCK_MHZ] =
            (unsigned long long)(clock64() - c.c0) * 1000ull / (global_ns() - c.t0 + 1);
      }
    }
  }
  __syncthreads();
  if (c.tid == 0) {
    const uint32_t prev = atomicAdd(&p.ctrl[CTRL_EXIT], 1u);
    if (prev == gridDim.x - 1) {
      p.ctrl[CTRL_EXIT] = 0u;
      *reinterpret_cast<unsigned long long*>(p.ctrl + CTRL_UCOUNT) = 0ull;
      uint32_t e = p.ctrl[CTRL_EPOCH] + 1u;
      if (e == 0xffffffffu) e = 0u;
      p.ctrl[CTRL_EPOCH] = e;
    }
  }
}

}  // namespace moe
