// The expert-range single kernel of the MoE decode layer step (sm_103a).
//
// Each CTA owns contiguous ranges of the step's work instead of a share of every
// expert:
//   gate/up  a contiguous range of the (routed slot u, intermediate row j) items,
//            u-major, split over the CTAs by cost -- at M = 1 the 8 x 768 rows
//            of Ling's routed experts are 40 or 41 rows per CTA, so a CTA touches
//            one or two experts;
//   down     a contiguous range of the (routed slot u, output block b) stages,
//            b over the grid's output blocks of H / grid rows -- at M = 1 each CTA
//            takes 8 blocks (135 rows) of one or two experts, the same experts its
//            gate/up range covered;
//   shared   every CTA computes a 1/grid share of the shared expert's rows before
//            routing is known, and the shared expert's down rows of its own block.
// A down stage needs its expert's whole h (all I rows), which ~19 CTAs produce:
// per slot, a publisher warp counts the CTA's stored h rows with one fence and a
// count, and a fetcher warp copies the slot's h into shared memory once the count
// reaches I. Nothing else waits on other CTAs after routing: each CTA streams
// its ~0.6 MB (M = 1) back to back, and the ring keeps streaming down weights
// while the h of their slot is still on its way.
//
// The combine (Ling-3.0-flash batch-1 decode blog, section "PDL: stacking the
// latency floors of small kernels": one fp32 sum, one final cast): every down
// stage stores its rows' fp32 results per (output block, slot, token row) in
// global memory as run-tagged 64-bit words (run tag << 32 | value: the data is
// its own readiness flag, no fence -- "Muse Spark Open Ultrafast", section
// "Megakernel internals"); CTA b owns output block b and, after its own down
// stages, polls the block's words of every slot until all carry this run's tag,
// sums them in slot order, adds the residual and writes bf16 once.
//
// Code size matters here: the kernel runs once per layer step, so every
// instruction it executes is fetched again at each launch unless the SM's
// instruction cache holds the whole kernel. Loops are unrolled only where it
// feeds the FMA pipe.
#pragma once
#include "moe_kernels.cuh"

namespace moe {

constexpr int kDRowLanes = 16;                        // threads per down row
constexpr int kDRowsPass = kNC * 32 / kDRowLanes;     // down rows per pass (24)
constexpr int kDChunk = 8;                            // 16-byte chunks per thread and row (I <= 1024)

// The down segments of this CTA: the shared slot's block (S == 1), then the
// routed (slot, output block) stages of its range, grouped by slot.
struct FlatSegs {
  int n;
  int sl[kFlatSegs], b0[kFlatSegs], b1[kFlatSegs];
};

__device__ __forceinline__ FlatSegs flat_segs(const Params& p, int nrouted) {
  FlatSegs s;
  s.n = 0;
  if (p.S > 0) {
    s.sl[0] = 0;
    s.b0[0] = blockIdx.x;
    s.b1[0] = blockIdx.x + 1;
    s.n = 1;
  }
  int lo, hi;
  split_range(nrouted * p.grid, blockIdx.x, p.grid, lo, hi);
  while (lo < hi && s.n < kFlatSegs) {
    const int u = lo / p.grid;
    const int end = min(hi, (u + 1) * p.grid);
    s.sl[s.n] = p.S + u;
    s.b0[s.n] = lo - u * p.grid;
    s.b1[s.n] = end - u * p.grid;
    ++s.n;
    lo = end;
  }
  return s;
}

// First output row of block b (blocks split H over the grid).
__device__ __forceinline__ int flat_row(const Params& p, int b) {
  return (int)((unsigned)p.H * (unsigned)b / (unsigned)p.grid);
}

// Gate/up items [lo, hi) of the flattened (slot, row) sequence of slots slot0..,
// warps w0 .. w0 + nw - 1 taking them; every warp arrives on a slot's counter
// after its items of that slot (also when it had none).
template <int FMT, int MAXM>
__device__ __forceinline__ Ring flat_items(const Ctx& c, const Route& rt, int lo, int hi, int slot0, bool shared,
                                           Ring ring, int w0, int nw, int q) {
  const Params& p = c.p;
  int* acnt = reinterpret_cast<int*>(c.sm + p.off_acnt);
  const uint4* xs = reinterpret_cast<const uint4*>(c.sm + p.off_x);
  XRegs<FMT, MAXM> xr;
  load_xregs<FMT, MAXM>(c, xr);
  ItemWalk w(lo, hi, q, p.I);
  w.w0 = w0;
  w.nw = nw;
  int cur = lo < hi ? w.u : -1;
  auto arrive = [&](int sl) {
    fence_proxy_async_global();  // the h stores are read by other CTAs' bulk copies
    __syncwarp();
    if (c.lane == 0) {
      __threadfence_block();
      atomicAdd(acnt + sl, 1);
    }
  };
#pragma unroll 1
  for (; w.more(); ring.next(p.nslots)) {
    if (w.u != cur) {
      arrive(cur + slot0);
      cur = w.u;
    }
    item_stage<FMT, MAXM>(c, rt, w, ring, w.u + slot0, shared, xr, xs, false);
    w.advance(w.count());
  }
  if (cur >= 0) arrive(cur + slot0);
  return ring;
}

// Output block of row o (blocks split H over the grid: block b starts at
// floor(H b / grid)).
__device__ __forceinline__ int flat_block(const Params& p, int o) {
  return (int)(((unsigned)(o + 1) * (unsigned)p.grid - 1u) / (unsigned)p.H);
}

// One down stage: rows [0, nr) of the stage (W2 rows o = R0 + r of one expert)
// against the slot's h (hs: the slot's pairs in ascending row order); the fp32
// sums are stored tagged to the owner block's words (rows that did not choose
// the expert store a tagged zero, so the owner finds every word of the run).
// 16 threads per row, each with chunks sub, sub + 16, ... of the row; every lane
// of a warp runs the same number of passes (rows past nr repeat the last one and
// are not stored), so the 16-lane reductions stay converged.
template <int MAXM>
__device__ __forceinline__ void flat_down_stage(const Params& p, const uint8_t* st, int nr, const float* hs,
                                                uint32_t mask, const float (&hr)[kDChunk][8], int sl, int R0,
                                                uint32_t ep, int tid) {
  const int sub = tid & (kDRowLanes - 1);
  const int nch = p.nchunk_i;
#pragma unroll 1
  for (int r0 = (tid >> 5) * 2; r0 < nr; r0 += kDRowsPass) {
    const int r = r0 + ((tid >> 4) & 1);
    const uint4* wr = reinterpret_cast<const uint4*>(st + (size_t)min(r, nr - 1) * p.row2);
    float acc[MAXM];
#pragma unroll
    for (int m = 0; m < MAXM; ++m) acc[m] = 0.0f;
#pragma unroll
    for (int k = 0; k < kDChunk; ++k) {
      const int ch = sub + kDRowLanes * k;
      if (ch < nch) {
        const uint4 wv = wr[ch];
        if (MAXM == 1) {
          dot8_bf16_f32(acc[0], wv, hr[k]);
        } else {
          int hp = 0;
#pragma unroll
          for (int m = 0; m < MAXM; ++m) {
            if (mask >> m & 1u) {
              const float4* h4 = reinterpret_cast<const float4*>(hs + (size_t)hp * p.I + 8 * ch);
              const float4 a = h4[0], b = h4[1];
              const float hv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
              dot8_bf16_f32(acc[m], wv, hv);
              ++hp;
            }
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MAXM; ++m)
#pragma unroll
      for (int o = kDRowLanes / 2; o; o >>= 1) acc[m] += __shfl_xor_sync(kFull, acc[m], o);
    if (sub == 0 && r < nr) {
      const int o = R0 + r, b = flat_block(p, o);
      unsigned long long* y = p.ybuf + ((size_t)b * p.nslot_max + sl) * p.maxm * p.flat_rb + (o - flat_row(p, b));
#pragma unroll
      for (int m = 0; m < MAXM; ++m)
        if (m < p.M) st_tagged(y + (size_t)m * p.flat_rb, ep, (mask >> m & 1u) ? acc[m] : 0.0f);
    }
  }
}

// The down phase of the consumers: every segment's stages in ring order.
template <int MAXM>
__device__ __forceinline__ Ring flat_down(const Ctx& c, const Route& rt, const FlatSegs& sg, Ring ring) {
  const Params& p = c.p;
  const uint32_t hbar0 = smem_u32(c.sm + p.off_hbar);
  const int drs = p.d_rows_stage;
#pragma unroll
  for (int k = 0; k < kFlatSegs; ++k) {  // unrolled: the segment table stays in registers
    if (k >= sg.n) break;
    const int sl = sg.sl[k];
    const uint32_t mask = rt.slot_mask[sl];
    const float* hs = reinterpret_cast<const float*>(c.sm + p.off_hs) + (size_t)k * p.maxm * p.I;
    const bool have = !c.aborted() && c.wait_bar(hbar0 + 8u * k, 0, SITE_HIDDEN);
    float hr[kDChunk][8];
    if (MAXM == 1 && have) {
      const int sub = c.tid & (kDRowLanes - 1);
#pragma unroll
      for (int kk = 0; kk < kDChunk; ++kk) {
        const int ch = sub + kDRowLanes * kk;
        if (ch < p.nchunk_i) {
          const float4 a = *reinterpret_cast<const float4*>(hs + 8 * ch);
          const float4 b = *reinterpret_cast<const float4*>(hs + 8 * ch + 4);
          hr[kk][0] = a.x; hr[kk][1] = a.y; hr[kk][2] = a.z; hr[kk][3] = a.w;
          hr[kk][4] = b.x; hr[kk][5] = b.y; hr[kk][6] = b.z; hr[kk][7] = b.w;
        }
      }
    }
    if (k == 0 && c.tid == 0) c.stamp(ST_D_FIRST);
    const int R1 = flat_row(p, sg.b1[k]);
#pragma unroll 1
    for (int r0 = flat_row(p, sg.b0[k]); r0 < R1; r0 += drs, ring.next(p.nslots)) {
      const int nr = min(drs, R1 - r0);
      const bool got = !c.aborted() && c.wait_full(ring);
      if (got && have)
        flat_down_stage<MAXM>(p, c.slot_ptr(ring.slot), nr, hs, mask, hr, sl, r0, c.epoch(), c.tid);
      __syncwarp();
      if (got && c.lane == 0) c.release(ring, 1);
    }
  }
  return ring;
}

// After its own down stages, CTA b finishes output block b: it polls the block's
// tagged words of every slot (bounded) until all carry this run's tag, then sums
// each output row over the slots in slot order, adds the residual and writes
// bf16 with one rounding.
template <int MAXM>
__device__ __forceinline__ void flat_finish(const Ctx& c, int nsl) {
  const Params& p = c.p;
  const int b = blockIdx.x, o0 = flat_row(p, b), nr = flat_row(p, b + 1) - o0;
  if (nr == 0) return;
  float* stg = reinterpret_cast<float*>(c.sm + p.off_ring);  // the ring is idle now: [slot][row m][nr]
  const uint32_t ep = c.epoch();
  const unsigned long long* yb = p.ybuf + (size_t)b * p.nslot_max * p.maxm * p.flat_rb;
  const int n = nsl * p.M * nr;
  const int nthr = kNC * 32;
  uint32_t spins = 0;
  bool ok = !c.aborted();
  for (int base = c.tid; ok && base < n; base += nthr * kStageBatch) {
    uint32_t pending = 0;
#pragma unroll
    for (int k = 0; k < kStageBatch; ++k)
      if (base + k * nthr < n) pending |= 1u << k;
    while (pending) {
      unsigned long long v[kStageBatch];
#pragma unroll
      for (int k = 0; k < kStageBatch; ++k) {
        v[k] = 0;
        const int i = base + k * nthr;
        if (pending >> k & 1u) {
          const int sl = i / (p.M * nr), m = (i / nr) % p.M, j = i % nr;
          v[k] = ld_relaxed_u64(yb + ((size_t)sl * p.maxm + m) * p.flat_rb + j);
        }
      }
#pragma unroll
      for (int k = 0; k < kStageBatch; ++k) {
        if ((pending >> k & 1u) && (uint32_t)(v[k] >> 32) == ep) {
          stg[base + k * nthr] = __uint_as_float((uint32_t)v[k]);
          pending &= ~(1u << k);
        }
      }
      if (!pending) break;
      __nanosleep(32);
      if ((++spins & 15) == 0) {
        if (c.aborted() || c.peer_failed()) {
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
  if (p.out_aliases_x && ok) wait_xflags(c);
  bar_sync(kBarConsumers, kNC * 32);
  if (c.aborted()) return;
  for (int i = c.tid; i < p.M * nr; i += nthr) {
    const int m = i / nr, j = i % nr;
    float y = 0.0f;
    for (int sl = 0; sl < nsl; ++sl) y += stg[((size_t)sl * p.M + m) * nr + j];  // zeros where row m has no value
    const size_t at = (size_t)m * p.H + o0 + j;
    const float rv = __uint_as_float((uint32_t)p.resid[at] << 16);
    p.out[at] = f32_to_bf16_bits(rv + y);
  }
}

// The publisher (lane 0 of its warp): once every consumer warp has arrived on a
// slot of this CTA's gate/up ranges, one fence releases the CTA's h stores of all
// slots found complete, and the slot counts grow by the CTA's rows of them.
__device__ __forceinline__ void flat_publish(const Ctx& c) {
  const Params& p = c.p;
  volatile int* acnt = reinterpret_cast<volatile int*>(c.sm + p.off_acnt);
  // entries: the shared slot's share, then each routed slot of [ULO, UHI)
  int slo, shi;
  split_range(p.S * p.I, blockIdx.x, p.grid, slo, shi);
  const int ulo = c.misc[MISC_ULO], uhi = c.misc[MISC_UHI];
  const int n_sh = shi > slo ? 1 : 0;
  const int u0 = ulo / p.I;
  const int n_ro = uhi > ulo ? (uhi - 1) / p.I - u0 + 1 : 0;
  auto entry = [&](int i, int& sl, int& cnt) {
    if (i < n_sh) {
      sl = 0;
      cnt = shi - slo;
    } else {
      const int u = u0 + i - n_sh;
      sl = p.S + u;
      cnt = min(uhi, (u + 1) * p.I) - max(ulo, u * p.I);
    }
  };
  const int n = n_sh + n_ro;
  uint32_t spins = 0;
  for (int pub = 0; pub < n;) {
    int np = pub;
    for (;;) {
      if (np >= n) break;
      int sl, cnt;
      entry(np, sl, cnt);
      if (acnt[sl] < kNC) break;
      ++np;
    }
    if (np > pub) {
      __threadfence();  // acquires the warps' h stores (through the counters) and releases them
      for (; pub < np; ++pub) {
        int sl, cnt;
        entry(pub, sl, cnt);
        red_add_u32(p.ctrl + CTRL_SLOTCNT + sl, (uint32_t)cnt);
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

// The fetcher (lane 0 of its warp): each down segment's h (the slot's pairs, all
// I values) into its shared-memory buffer as soon as every CTA has counted the
// slot, counted on the segment's mbarrier.
__device__ __forceinline__ void flat_fetch(const Ctx& c, const Route& rt, const FlatSegs& sg) {
  const Params& p = c.p;
  const uint32_t hbar0 = smem_u32(c.sm + p.off_hbar);
  const float* rep = p.hbuf + (size_t)(blockIdx.x % kHRep) * p.npair_max * p.I;
  int issued = 0;
  uint32_t spins = 0;
#pragma unroll
  for (int k = 0; k < kFlatSegs; ++k) {
    if (k >= sg.n || c.aborted()) break;
    const int sl = sg.sl[k];
    while (ld_acquire_u32(p.ctrl + CTRL_SLOTCNT + sl) < (uint32_t)p.I) {
      __nanosleep(32);
      if ((++spins & 15) == 0) {
        if (c.aborted()) break;
        if (c.peer_failed()) {
          c.abort_local();
          break;
        }
        if (c.expired()) {
          c.fail(SITE_HIDDEN);
          break;
        }
      }
    }
    if (c.aborted()) break;
    fence_proxy_async_global();  // the acquired h stores before the bulk copy that reads them
    const int p0 = rt.pair_base[sl];
    const uint32_t bytes = (uint32_t)(rt.pair_base[sl + 1] - p0) * (uint32_t)p.I * 4u;
    float* dst = reinterpret_cast<float*>(c.sm + p.off_hs) + (size_t)k * p.maxm * p.I;
    mbar_arrive_expect_tx(hbar0 + 8u * k, bytes);
    bulk_g2s_plain(smem_u32(dst), rep + (size_t)p0 * p.I, bytes, hbar0 + 8u * k);
    ++issued;
  }
  // copies issued but not waited for by the consumers (after an abort) land before exit
  if (c.aborted()) {
    const uint64_t t = global_ns();
    for (int k = 0; k < issued; ++k)
      while (!mbar_try_wait(hbar0 + 8u * k, 0) && global_ns() - t < p.timeout_ns) {
      }
  }
}

// The producer's stage sequence (lane 0): x, router rows, the shared expert's
// gate/up rows of this CTA's share, [routing], the routed gate/up rows of the
// CTA's range, then every down segment's W2 rows.
__device__ __forceinline__ void flat_produce_pairs(Producer& pr, const Route& rt, int lo, int hi, int q, bool shared) {
  const Params& p = pr.c.p;
  for (ItemWalk w(lo, hi, q, p.I); w.more(); pr.ring.next(p.nslots)) {
    const int nq = w.count();
    uint32_t dst, bar;
    if (!pr.begin((uint32_t)nq * p.pair_bytes, dst, bar)) return;
    pr.copy_pairs(shared ? -1 - w.u : rt.slot_e[p.S + w.u], w.j, nq, dst, bar);
    w.advance(nq);
  }
}

__device__ __forceinline__ void flat_produce_down(Producer& pr, const Route& rt, const FlatSegs& sg) {
  const Params& p = pr.c.p;
#pragma unroll
  for (int k = 0; k < kFlatSegs; ++k) {
    if (k >= sg.n) break;
    const int sl = sg.sl[k];
    const int e = sl < p.S ? -1 - sl : rt.slot_e[sl];
    const uint8_t* wt = e >= 0 ? p.w2 : p.sh_w2;
    const size_t ex = (size_t)(e >= 0 ? e : -1 - e);
    const int R1 = flat_row(p, sg.b1[k]);
    for (int r0 = flat_row(p, sg.b0[k]); r0 < R1; r0 += p.d_rows_stage, pr.ring.next(p.nslots)) {
      const uint32_t bytes = (uint32_t)min(p.d_rows_stage, R1 - r0) * p.row2;
      uint32_t dst, bar;
      if (!pr.begin(bytes, dst, bar)) return;
      bulk_g2s(dst, wt + (ex * p.H + r0) * p.row2, bytes, bar, pr.pol);
    }
  }
}

template <int FMT, int MAXM>
__global__ void __launch_bounds__(kThreadsFlat, 1) moe_flat_kernel(const __grid_constant__ Params p) {
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
    for (int k = 0; k < kFlatSegs; ++k) mbar_init(smem_u32(sm + p.off_hbar) + 8u * k, 1);
    mbar_init_fence();
    c.misc[MISC_ABORT] = 0;
    c.misc[MISC_NROUTED] = 0;
    c.misc[MISC_ROUTED] = 0;
  }
  for (int i = c.tid; i < p.nslot_max; i += kThreadsFlat) reinterpret_cast<int*>(sm + p.off_acnt)[i] = 0;
  for (int e = c.tid; e < p.E; e += kThreadsFlat) rt.emask[e] = 0u;
  for (int e = c.tid; e < (p.E + 31) / 32; e += kThreadsFlat) rt.bitmap[e] = 0u;
  __syncthreads();

  if (c.warp > kNC) {
    // ------------------------------------------------------------ hand-off warps
    __syncwarp();
    bar_sync(kBarRoute, kThreadsFlat);
    if (c.lane == 0) {
      if (c.warp == kNC + 1) {
        flat_publish(c);
      } else {
        const FlatSegs sg = flat_segs(p, c.misc[MISC_NROUTED]);
        flat_fetch(c, rt, sg);
      }
    }
    __syncwarp();
  } else if (c.warp == kNC) {
    // ------------------------------------------------------------ producer
    Producer pr(c);
    int slo, shi;
    split_range(p.S * p.I, blockIdx.x, p.grid, slo, shi);
    if (c.lane == 0) {
      c.stamp(ST_START);
      pr.x_rows();
      pr.router();
      flat_produce_pairs(pr, rt, slo, shi, p.q, true);
      c.stamp(ST_P_R_ISSUED);
    }
    __syncwarp();
    bar_sync(kBarRoute, kThreadsFlat);
    if (c.lane == 0) {
      c.stamp(ST_P_ROUTE);
      const FlatSegs sg = flat_segs(p, c.misc[MISC_NROUTED]);
      flat_produce_pairs(pr, rt, c.misc[MISC_ULO], c.misc[MISC_UHI], p.q, false);
      c.stamp(ST_P_U_ISSUED);
      flat_produce_down(pr, rt, sg);
      c.stamp(ST_P_D_ISSUED);
      if (c.aborted()) {
        pr.drain();
        // the x copy may still be in flight if the consumers gave up before it landed
        const uint64_t t = global_ns();
        while (!mbar_try_wait(c.xbar, 0) && global_ns() - t < p.timeout_ns) {
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    if (c.tid == 0) c.misc[MISC_EPOCH] = (int)ld_relaxed_u32(&p.ctrl[CTRL_EPOCH]);
    prepare_x(c);
    bar_sync(kBarConsumers, kNC * 32);
    if (c.tid == 0) c.stamp(ST_X_LOADED);
    if (p.out_aliases_x && c.tid == 0) st_tagged(p.xflags + blockIdx.x, c.epoch(), 0.0f);
    Ring ring;
    ring = consume_router<MAXM>(c, ring);
    bar_sync(kBarConsumers, kNC * 32);  // this CTA's logits are all stored
    if (c.tid == 0) {
      c.stamp(ST_RFLAG);
    }
    // every consumer warp routes (the logits staged by all of them, each row's
    // top-k spread over several warps); the shared expert's items follow
    route_rows<MAXM>(c, rt, true, kNC * 32, kBarRouting);
    fence_proxy_async_shared();  // the routing scratch becomes the h buffers (bulk copies)
    if (c.tid == 0) reinterpret_cast<volatile int*>(c.misc)[MISC_ROUTED] = 1;  // hint for the producer's prefetch
    bar_arrive(kBarRoute, kThreadsFlat);
    if (c.tid == 0) c.stamp(ST_ROUTED);
    int slo, shi;
    split_range(p.S * p.I, blockIdx.x, p.grid, slo, shi);
    ring = flat_items<FMT, MAXM>(c, rt, slo, shi, 0, true, ring, 0, kNC, p.q);
    if (c.tid == 0) c.stamp(ST_R_DONE);
    const int nrouted = c.misc[MISC_NROUTED];
    ring = flat_items<FMT, MAXM>(c, rt, c.misc[MISC_ULO], c.misc[MISC_UHI], p.S, false, ring, 0, kNC, p.q);
    if (c.tid == 0) c.stamp(ST_U_DONE);
    const FlatSegs sg = flat_segs(p, nrouted);
    ring = flat_down<MAXM>(c, rt, sg, ring);
    if (c.tid == 0) c.stamp(ST_D_SUMMED);
    bar_sync(kBarConsumers, kNC * 32);  // every consumer is done with the ring
    flat_finish<MAXM>(c, p.S + nrouted);
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
      for (int i = 0; i < p.nslot_max; ++i) p.ctrl[CTRL_SLOTCNT + i] = 0u;
      uint32_t e = p.ctrl[CTRL_EPOCH] + 1u;
      if (e == 0xffffffffu) e = 0u;
      p.ctrl[CTRL_EPOCH] = e;
    }
  }
}

}  // namespace moe
