// C ABI of the MoE decode layer step: config validation, launch planning,
// scratch ownership and kernel launches. See include/moe_decode.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include "../../include/moe_decode.h"
#include "internal.h"
#include "kernel_table.h"
#include "moe_params.h"

using moe::Params;

struct moe_decode_handle {
  moe_decode_config cfg;
  Params base;       // everything but the per-run pointers and M
  Params ilv;        // the same for the slot-interleaved single kernel (when has_ilv)
  Params flat;       // the same for the expert-range single kernel (when has_flat)
  bool has_ilv = false;
  bool has_flat = false;
  bool sk = false;    // down matrices transposed: the split-K single kernel only
  int ilv_mode = 1;   // MOE_OPT_INTERLEAVE
  int flat_mode = 0;  // MOE_OPT_FLAT
  int device = 0;
  int sched = MOE_SCHED_PERSISTENT;
  int max_slots = 0;  // ring slots the planned shared memory holds
  int max_slots_ilv = 0;
  int max_slots_flat = 0;
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  uint16_t* stage_x = nullptr;  // run_host staging
  uint16_t* stage_r = nullptr;
  uint16_t* stage_out = nullptr;
  int32_t* stage_idx = nullptr;
  float* stage_w = nullptr;
  // run_host read-back: the device block [status words .. top-k .. output rows]
  // (contiguous after the control words) and its pinned host copy
  uint8_t* host_rb = nullptr;
  size_t rb_si = 0, rb_sw = 0, rb_so = 0;  // byte offsets of topk_idx, topk_w, out in the block
};

namespace {

constexpr unsigned long long kDefaultTimeoutNs = 1000000000ull;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

moe_status check_config(const moe_decode_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  const int H = c->hidden, I = c->inter, E = c->num_experts, K = c->top_k;
  if (H <= 0 || I <= 0 || E <= 0 || K <= 0 || c->num_shared < 0 || c->max_rows <= 0)
    return MOE_ERR_INVALID_ARG;
  if (c->score != MOE_SCORE_SOFTMAX_TOPK_RENORM && c->score != MOE_SCORE_SIGMOID_BIAS) return MOE_ERR_UNSUPPORTED;
  if (c->sched < MOE_SCHED_PERSISTENT || c->sched > MOE_SCHED_CHAIN) return MOE_ERR_UNSUPPORTED;
  if (E < 2 || E > 1024 || (E & 1)) return MOE_ERR_UNSUPPORTED;
  if (K > 16 || K > E) return MOE_ERR_UNSUPPORTED;
  if (c->num_shared > 4 || c->max_rows > moe::kMaxRowsRun) return MOE_ERR_UNSUPPORTED;
  if (!std::isfinite(c->routed_scale)) return MOE_ERR_INVALID_ARG;
  if (c->pre_rmsnorm && !(c->rms_eps > 0.0f && std::isfinite(c->rms_eps))) return MOE_ERR_INVALID_ARG;
  if (c->w2_layout != MOE_W2_H_I && c->w2_layout != MOE_W2_I_H) return MOE_ERR_UNSUPPORTED;
  if (c->w2_layout == MOE_W2_I_H) {
    // the split-K kernel: every output column of the transposed down rows to one
    // consumer thread (8 per thread), one persistent kernel
    if (c->sched != MOE_SCHED_PERSISTENT || H / 8 > moe::kNC * 32) return MOE_ERR_UNSUPPORTED;
    if (c->wdtype == MOE_W_BF16) {
      if (H % 8 || H < 64 || I % 8) return MOE_ERR_UNSUPPORTED;
    } else if (c->wdtype == MOE_W_FP8_BLOCK) {
      if (H % moe::kFp8Block || I % moe::kFp8Block) return MOE_ERR_UNSUPPORTED;
    } else {
      return MOE_ERR_UNSUPPORTED;
    }
    return MOE_OK;
  }
  if (c->wdtype == MOE_W_BF16) {
    if (H % 8 || H < 64 || H > 4096) return MOE_ERR_UNSUPPORTED;
    const int tg = I / 8;
    if (I % 8) return MOE_ERR_UNSUPPORTED;
    if (!((tg <= 32 && pow2(tg)) || (tg % 32 == 0 && tg <= moe::kNC * 32))) return MOE_ERR_UNSUPPORTED;
  } else if (c->wdtype == MOE_W_NVFP4) {
    if (H % 256 || H < 256 || H > 4096) return MOE_ERR_UNSUPPORTED;
    if (I % 256 || I / 32 > moe::kNC * 32) return MOE_ERR_UNSUPPORTED;
  } else if (c->wdtype == MOE_W_FP8_BLOCK) {
    // 128 x 128 scale blocks; 8-code down chunks, I / 8 threads per down row as bf16
    if (H % moe::kFp8Block || H > 4096 || I % moe::kFp8Block) return MOE_ERR_UNSUPPORTED;
    const int tg = I / 8;
    if (!((tg <= 32 && pow2(tg)) || (tg % 32 == 0 && tg <= moe::kNC * 32))) return MOE_ERR_UNSUPPORTED;
  } else {
    return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

// Plans the per-CTA layout for a device with `sms` SMs and `smem_optin` bytes
// of opt-in shared memory per block.
// ilv: the layout of the slot-interleaved single kernel (every output row of a
// CTA in one down stage, whose ring slot also holds the slot's h rows; no h
// staging area). MOE_ERR_UNSUPPORTED when that layout does not fit.
moe_status plan(const moe_decode_config& c, int sms, int smem_optin, Params& p, bool ilv) {
  std::memset(&p, 0, sizeof(p));
  const int H = c.hidden, I = c.inter, E = c.num_experts, K = c.top_k, S = c.num_shared;
  // one launch handles at most kMaxRowsLaunch rows; a run of more splits into launches
  const int maxm = std::min(c.max_rows, moe::kMaxRowsLaunch);
  p.H = H; p.I = I; p.E = E; p.K = K; p.S = S; p.maxm = maxm;
  p.fmt = c.wdtype == MOE_W_BF16 ? moe::FMT_BF16 : c.wdtype == MOE_W_NVFP4 ? moe::FMT_NVFP4 : moe::FMT_FP8;
  p.score = c.score == MOE_SCORE_SIGMOID_BIAS ? 1 : 0;
  p.routed_scale = c.routed_scale;
  p.rms_eps = c.rms_eps;
  p.pre_rmsnorm = c.pre_rmsnorm ? 1 : 0;
  if (p.fmt == moe::FMT_BF16) {
    p.nchunk_h = H / 8; p.row13 = 2 * H; p.sc13 = 0;
    p.nchunk_i = I / 8; p.row2 = 2 * I; p.sc2 = 0;
  } else if (p.fmt == moe::FMT_FP8) {  // block scales are read by the consumers, not staged
    p.nchunk_h = H / 16; p.row13 = H; p.sc13 = 0;
    p.nchunk_i = I / 8; p.row2 = I; p.sc2 = 0;
  } else {
    p.nchunk_h = H / 32; p.row13 = H / 2; p.sc13 = H / 16;
    p.nchunk_i = I / 32; p.row2 = I / 2; p.sc2 = I / 16;
  }
  p.tg = p.nchunk_i;
  p.ng = moe::kNC * 32 / p.tg;
  p.pair_bytes = 2 * (p.row13 + p.sc13);
  if (p.fmt == moe::FMT_FP8) {
    // the expert's whole block-scale matrix rides behind each of its stages (bulk
    // copies need multiples of 16 bytes; else the consumers read them from global)
    const size_t s13 = (size_t)(2 * I / moe::kFp8Block) * (H / moe::kFp8Block) * 4;
    const size_t s2 = (size_t)(H / moe::kFp8Block) * (I / moe::kFp8Block) * 4;
    p.sc13e = (s13 % 16 == 0 && s13 <= (size_t)moe::kFp8StagedScaleMax) ? (int)s13 : 0;
    p.sc2e = (s2 % 16 == 0 && s2 <= (size_t)moe::kFp8StagedScaleMax) ? (int)s2 : 0;
  }
  p.rpair_bytes = 4 * H;
  p.grid = sms;
  p.nslot_max = S + std::min(E, maxm * K);
  p.npair_max = S * maxm + maxm * K;
  // fixed shared-memory blocks
  size_t off = 0;
  auto take = [&](size_t bytes, size_t align) {
    off = round_up(off, align);
    const size_t at = off;
    off += bytes;
    return static_cast<int>(at);
  };
  p.off_full = take(moe::kMaxSlots * 8, 8);
  p.off_empty = take(moe::kMaxSlots * 8, 8);
  p.off_xbar = take(8, 8);
  p.off_xfree = take(8, 8);
  p.off_hbar = take(16, 8);
  p.off_slot_seq = take(moe::kMaxSlots * 4, 4);
  p.off_x = take((size_t)maxm * H * 2, 128);
  p.off_sel_e = take(((size_t)maxm * K * 4 + 15) / 16 * 16 + 16, 16);  // read in 16-byte groups by the one-row union
  p.off_sel_w = take((size_t)maxm * K * 4, 4);
  p.off_emask = take((size_t)E * 4, 4);
  p.off_bitmap = take((size_t)(E + 31) / 32 * 4, 4);
  p.off_slot_of = take((size_t)E * 4, 4);
  p.off_slot_e = take((size_t)p.nslot_max * 4, 4);
  p.off_slot_mask = take((size_t)p.nslot_max * 4, 4);
  p.off_slot_w = take((size_t)p.nslot_max * maxm * 4, 4);
  p.off_pair_base = take((size_t)(p.nslot_max + 1) * 4, 4);
  p.off_pair_sr = take((size_t)p.npair_max * 4, 4);
  p.off_red = take((size_t)moe::kNC * moe::kRpgMax * 8 * 4, 16);
  p.off_misc = take(moe::MISC_WORDS * 4, 16);
  p.off_ucnt = take(moe::ILV_WORDS * 4, 16);
  p.off_dslot = take((size_t)p.nslot_max * 4, 4);
  p.off_bias = p.score ? take((size_t)E * 4, 16) : 0;
  const size_t fixed = round_up(off, 128);
  const long long avail = (long long)smem_optin - 1024 - (long long)fixed;
  // ring slot: one stage of ~kStageTarget bytes, at least one router pair, one
  // gate/up pair and one down stage of this CTA's rows
  const int rows_per_cta = (H + p.grid - 1) / p.grid;
  int drs = std::min(rows_per_cta, moe::rows_per_group(p.fmt) * p.ng);
  if (ilv) {
    // every output row of the CTA in one down stage, then the slot's h rows
    // (at most maxm pairs); the counters hold every union slot
    if (drs < rows_per_cta || p.nslot_max > moe::CTRL_WORDS - moe::CTRL_SLOTCNT) return MOE_ERR_UNSUPPORTED;
    p.d_soff = (int)round_up((size_t)drs * (p.row2 + p.sc2), 16);
    p.d_hoff = (int)round_up((size_t)p.d_soff + p.sc2e, 16);
  }
  // a slot holds a whole number of gate/up pairs (about kStageTarget bytes), so
  // that no slot space is left unused in the gate/up phases
  const size_t q0 = std::max<size_t>(1, std::min<size_t>(moe::kNC, moe::kStageTarget / p.pair_bytes));
  size_t slot = 0;
  for (;;) {
    const size_t dstage = ilv ? (size_t)p.d_hoff + (size_t)maxm * I * 4
                              : round_up((size_t)drs * (p.row2 + p.sc2), 16) + p.sc2e;
    slot = round_up(std::max({q0 * p.pair_bytes + p.sc13e, (size_t)p.rpair_bytes, (size_t)p.pair_bytes + p.sc13e,
                              dstage}),
                    128);
    if (ilv || (long long)(moe::kMinSlots * slot) <= avail - (long long)maxm * I * 4 || drs == 1) break;
    drs = (drs + 1) / 2;
  }
  // h staging area: all (expert, row) pairs when they fit next to kMinSlots ring
  // slots, else as many as fit (at least one slot's worth: maxm rows)
  const size_t per_pair = (size_t)I * 4;
  long long hs_room = avail - (long long)(moe::kMinSlots * slot);
  int hs_pairs = (int)std::min<long long>(p.npair_max, hs_room > 0 ? hs_room / (long long)per_pair : 0);
  if (hs_pairs < maxm) hs_pairs = maxm;
  if (ilv) hs_pairs = 0;  // h rows travel in the down stages
  p.hs_pairs = hs_pairs;
  // all pairs at once; else two buffers (one batch lands while the other is in
  // use) when each holds a full slot's rows; else one buffer
  p.hs_nbuf = (!ilv && hs_pairs < p.npair_max && hs_pairs >= 2 * maxm) ? 2 : 1;
  p.off_hs = (int)fixed;
  // routing scratch shares the h staging area (routing is over before any h is staged)
  size_t ro = fixed;
  auto rtake = [&](size_t bytes, size_t align) {
    ro = round_up(ro, align);
    const size_t at = ro;
    ro += bytes;
    return static_cast<int>(at);
  };
  p.off_lg = rtake((size_t)maxm * E * 4, 16);
  p.off_cand = rtake((size_t)maxm * moe::kCandMax * 8, 16);
  p.off_lmax = rtake((size_t)maxm * 32 * 4, 16);
  p.off_thr = rtake((size_t)maxm * 8, 8);
  p.off_ccount = rtake((size_t)maxm * 4, 4);
  p.off_wtmp = rtake((size_t)maxm * 16 * 4, 16);
  p.off_wpc = rtake(32 * 4, 16);
  const size_t area = std::max(ro, fixed + (size_t)hs_pairs * per_pair);
  p.off_ring = (int)round_up(area, 128);
  const long long ring_budget = (long long)smem_optin - 1024 - p.off_ring;
  const long long ns = ring_budget > 0 ? ring_budget / (long long)slot : 0;
  if (ns < (ilv ? 3 : 2)) return MOE_ERR_UNSUPPORTED;
  p.slot_bytes = (int)slot;
  p.nslots = (int)std::min<long long>(ns, moe::kMaxSlots);
  // the h area is idle from the end of routing until the down phase: the routed
  // gate/up stages also use the slots that fit there
  // routed gate/up items are split by cost: streaming the pair plus the FMA work
  // of each row that chose the expert (fitted on GB300 per-CTA phase times: an
  // extra row adds ~1/6 of a bf16 item's time and about one NVFP4 item's)
  p.item_base = p.fmt == moe::FMT_BF16 ? 6 : p.fmt == moe::FMT_FP8 ? 3 : 1;
  p.off_xslot = (int)fixed;
  // the x rows are dead once the gate/up items are done: their area holds one
  // more down-phase slot when it is large enough
  // (it only ever takes down stages)
  const size_t dstage_bytes = round_up((size_t)drs * (p.row2 + p.sc2), 16) + p.sc2e;
  p.nslots_d = (!ilv && (size_t)maxm * H * 2 >= dstage_bytes && p.nslots < moe::kMaxSlots) ? 1 : 0;
  p.nslots_x = ilv ? 0 : (int)std::min<long long>((long long)(area - fixed) / (long long)slot, moe::kMaxSlots - p.nslots);
  // per-slot h fetches: measured faster for NVFP4 (its gate/up phase ends less
  // evenly across CTAs), not for bf16, which keeps one fetch after all h is stored.
  // Their mbarriers follow every ring slot's full barrier.
  p.hs_perslot = (!ilv && p.fmt == moe::FMT_NVFP4 && p.hs_nbuf == 1 && hs_pairs >= p.npair_max &&
                  p.nslot_max <= moe::kMaxSlots - moe::kHSlotBar &&
                  p.nslots + std::max(p.nslots_x, p.nslots_d) <= moe::kHSlotBar)
                     ? 1
                     : 0;
  p.d_rows_stage = drs;
  if (!ilv) p.d_soff = (int)round_up((size_t)drs * (p.row2 + p.sc2), 16);
  p.q = std::max(1, std::min(moe::kNC, (p.slot_bytes - p.sc13e) / p.pair_bytes));
  // router stages: at most kNC / 2 row pairs, so every row gets at least one warp
  p.qr = std::max(1, std::min(moe::kNC / 2, p.slot_bytes / p.rpair_bytes));
  p.smem_bytes = p.off_ring + p.nslots * p.slot_bytes + 1024;
  p.ilv_lag = 5;
  p.timeout_ns = kDefaultTimeoutNs;
  return MOE_OK;
}

// The layout of the expert-range single kernel (moe_flat.cuh): the shape fields
// of plan(), then its own shared memory: three h buffers (one per down segment)
// that the routing scratch overlaps, and a ring of gate/up / down stages.
// MOE_ERR_UNSUPPORTED when the kernel does not cover cfg (bf16 weights, at most
// one shared expert, routed slots no more than the grid's CTAs, I <= 1024).
moe_status plan_flat(const moe_decode_config& c, int sms, int smem_optin, Params& p) {
  moe_status st = plan(c, sms, smem_optin, p, false);
  if (st != MOE_OK) return st;
  p.sc13e = p.sc2e = p.d_soff = 0;
  if (p.fmt != moe::FMT_BF16 || p.S > 1 || p.nslot_max - p.S > p.grid ||
      p.nslot_max > moe::CTRL_WORDS - moe::CTRL_SLOTCNT || p.nchunk_i > moe::kFlatMaxChunks)
    return MOE_ERR_UNSUPPORTED;
  const int H = p.H, I = p.I, E = p.E, K = p.K, maxm = p.maxm;
  size_t off = 0;
  auto take = [&](size_t bytes, size_t align) {
    off = round_up(off, align);
    const size_t at = off;
    off += bytes;
    return static_cast<int>(at);
  };
  p.off_full = take(moe::kMaxSlots * 8, 8);
  p.off_empty = take(moe::kMaxSlots * 8, 8);
  p.off_xbar = take(8, 8);
  p.off_hbar = take(moe::kFlatSegs * 8, 8);
  p.off_slot_seq = take(moe::kMaxSlots * 4, 4);
  p.off_x = take((size_t)maxm * H * 2, 128);
  p.off_sel_e = take(((size_t)maxm * K * 4 + 15) / 16 * 16 + 16, 16);  // read in 16-byte groups by the one-row union
  p.off_sel_w = take((size_t)maxm * K * 4, 4);
  p.off_emask = take((size_t)E * 4, 4);
  p.off_bitmap = take((size_t)(E + 31) / 32 * 4, 4);
  p.off_slot_of = take((size_t)E * 4, 4);
  p.off_slot_e = take((size_t)p.nslot_max * 4, 4);
  p.off_slot_mask = take((size_t)p.nslot_max * 4, 4);
  p.off_slot_w = take((size_t)p.nslot_max * maxm * 4, 4);
  p.off_pair_base = take((size_t)(p.nslot_max + 1) * 4, 4);
  p.off_pair_sr = take((size_t)p.npair_max * 4, 4);
  p.off_red = take((size_t)moe::kNC * 8 * 4, 16);
  p.off_misc = take(moe::MISC_WORDS * 4, 16);
  p.off_acnt = take((size_t)p.nslot_max * 4, 4);
  p.off_bias = p.score ? take((size_t)E * 4, 16) : 0;
  const size_t fixed = round_up(off, 128);
  // h buffers; the routing scratch overlaps them (routing is over before any h lands)
  p.off_hs = (int)fixed;
  const size_t hbytes = (size_t)moe::kFlatSegs * maxm * I * 4;
  size_t ro = fixed;
  auto rtake = [&](size_t bytes, size_t align) {
    ro = round_up(ro, align);
    const size_t at = ro;
    ro += bytes;
    return static_cast<int>(at);
  };
  p.off_lg = rtake((size_t)maxm * E * 4, 16);
  p.off_cand = rtake((size_t)maxm * moe::kCandMax * 8, 16);
  p.off_lmax = rtake((size_t)maxm * 32 * 4, 16);
  p.off_thr = rtake((size_t)maxm * 8, 8);
  p.off_ccount = rtake((size_t)maxm * 4, 4);
  p.off_wtmp = rtake((size_t)maxm * 16 * 4, 16);
  p.off_wpc = rtake(32 * 4, 16);
  p.off_ring = (int)round_up(std::max(ro, fixed + hbytes), 128);
  const size_t q0 = std::max<size_t>(1, std::min<size_t>(moe::kNC, moe::kStageTarget / p.pair_bytes));
  const size_t slot = round_up(std::max({q0 * p.pair_bytes, (size_t)p.rpair_bytes, (size_t)p.pair_bytes,
                                         (size_t)p.row2}), 128);
  const long long ring_budget = (long long)smem_optin - 1024 - p.off_ring;
  const long long ns = ring_budget > 0 ? ring_budget / (long long)slot : 0;
  if (ns < 3) return MOE_ERR_UNSUPPORTED;
  p.slot_bytes = (int)slot;
  p.nslots = (int)std::min<long long>(ns, moe::kMaxSlots);
  p.q = std::max(1, std::min(moe::kNC, p.slot_bytes / p.pair_bytes));
  p.qr = std::max(1, std::min(moe::kNC / 2, p.slot_bytes / p.rpair_bytes));
  p.d_rows_stage = p.slot_bytes / p.row2;
  // the final combine stages its block's (slot, row, output) values in the ring
  p.flat_rb = ((H + p.grid - 1) / p.grid + 1) / 2 * 2;
  if ((long long)p.nslots * p.slot_bytes / 4 < (long long)p.nslot_max * maxm * p.flat_rb) return MOE_ERR_UNSUPPORTED;
  p.nslots_x = p.nslots_d = p.hs_pairs = p.hs_perslot = 0;
  p.hs_nbuf = 1;
  p.smem_bytes = p.off_ring + p.nslots * p.slot_bytes + 1024;
  return MOE_OK;
}

// The layout of the split-K single kernel (moe_sk.cuh; down matrices stored
// transposed): the shape fields of plan(), then its own shared memory -- this
// CTA's h rows and their tags, the routing scratch (overlapping the h rows:
// routing is over before any is stored), and a ring of gate/up stages (q row
// pairs) and transposed-down stages (dq rows). At the end the ring holds the
// CTA's block of every CTA's partial sums. MOE_ERR_UNSUPPORTED when the kernel
// does not cover cfg (bf16 or FP8 weights, H <= 8 * kNC * 32).
moe_status plan_sk(const moe_decode_config& c, int sms, int smem_optin, Params& p) {
  moe_status st = plan(c, sms, smem_optin, p, false);
  if (st != MOE_OK) return st;
  p.sc13e = p.sc2e = p.d_soff = 0;  // this kernel reads the FP8 block scales from global memory
  if (p.fmt == moe::FMT_NVFP4 || p.H / 8 > moe::kNC * 32 || p.H % 8) return MOE_ERR_UNSUPPORTED;
  const int H = p.H, I = p.I, E = p.E, K = p.K, S = p.S, maxm = p.maxm, G = p.grid;
  p.w2t = 1;
  p.item_base = p.fmt == moe::FMT_BF16 ? 6 : 3;  // as the row-block schedules: cost of an item with N rows
  // h rows one CTA may hold: its share of the shared experts' rows plus the
  // largest routed share the cost split can give (items cost item_base + N with
  // 1 <= N <= maxm, so a share holds at most (base + maxm) / (base + 1) times the
  // average, plus the items cut at both ends)
  const long long base = p.item_base;
  const long long routed = (long long)std::min(E, maxm * K) * I;
  const long long tcost = routed * (base + maxm);
  p.sk_rows_max = (int)((long long)(S * I + G - 1) / G + ((tcost + G - 1) / G + base) / (base + 1) + 4);
  size_t off = 0;
  auto take = [&](size_t bytes, size_t align) {
    off = round_up(off, align);
    const size_t at = off;
    off += bytes;
    return static_cast<int>(at);
  };
  p.off_full = take(moe::kMaxSlots * 8, 8);
  p.off_empty = take(moe::kMaxSlots * 8, 8);
  p.off_xbar = take(8, 8);
  p.off_psb = take(8, 8);
  p.off_slot_seq = take(moe::kMaxSlots * 4, 4);
  p.off_x = take((size_t)maxm * H * 2, 128);
  p.off_sel_e = take(((size_t)maxm * K * 4 + 15) / 16 * 16 + 16, 16);  // read in 16-byte groups by the one-row union
  p.off_sel_w = take((size_t)maxm * K * 4, 4);
  p.off_emask = take((size_t)E * 4, 4);
  p.off_bitmap = take((size_t)(E + 31) / 32 * 4, 4);
  p.off_slot_of = take((size_t)E * 4, 4);
  p.off_slot_e = take((size_t)p.nslot_max * 4, 4);
  p.off_slot_mask = take((size_t)p.nslot_max * 4, 4);
  p.off_slot_w = take((size_t)p.nslot_max * maxm * 4, 4);
  p.off_pair_base = take((size_t)(p.nslot_max + 1) * 4, 4);
  p.off_pair_sr = take((size_t)p.npair_max * 4, 4);
  p.off_red = take((size_t)moe::kNC * 8 * 4, 16);  // the router's partial dot products
  p.off_misc = take(moe::MISC_WORDS * 4, 16);
  p.off_psum = take((size_t)moe::kNC * 32 * 4, 16);
  // offsets of the other kernels' areas, unused here
  p.off_xfree = p.off_hbar = p.off_ucnt = p.off_dslot = p.off_xslot = p.off_acnt = 0;
  p.off_htag = take((size_t)p.sk_rows_max * 4, 16);
  p.off_bias = p.score ? take((size_t)E * 4, 16) : 0;
  const size_t fixed = round_up(off, 128);
  p.off_hsk = (int)fixed;
  p.off_hs = (int)fixed;
  size_t ro = fixed;
  auto rtake = [&](size_t bytes, size_t align) {
    ro = round_up(ro, align);
    const size_t at = ro;
    ro += bytes;
    return static_cast<int>(at);
  };
  p.off_lg = rtake((size_t)maxm * E * 4, 16);
  p.off_cand = rtake((size_t)maxm * moe::kCandMax * 8, 16);
  p.off_lmax = rtake((size_t)maxm * 32 * 4, 16);
  p.off_thr = rtake((size_t)maxm * 8, 8);
  p.off_ccount = rtake((size_t)maxm * 4, 4);
  p.off_wtmp = rtake((size_t)maxm * 16 * 4, 16);
  p.off_wpc = rtake(32 * 4, 16);
  p.off_ring = (int)round_up(std::max(ro, fixed + (size_t)p.sk_rows_max * maxm * 4), 1024);
  const size_t rowt = (size_t)H * (p.fmt == moe::FMT_BF16 ? 2 : 1);  // one transposed down row
  const size_t q0 = std::max<size_t>(1, std::min<size_t>(moe::kNC, moe::kStageTarget / p.pair_bytes));
  const size_t slot = round_up(std::max({q0 * p.pair_bytes, (size_t)p.rpair_bytes, (size_t)p.pair_bytes, rowt}), 128);
  const long long ring_budget = (long long)smem_optin - 1024 - p.off_ring;
  const long long ns = ring_budget > 0 ? ring_budget / (long long)slot : 0;
  if (ns < 3) return MOE_ERR_UNSUPPORTED;
  p.slot_bytes = (int)slot;
  p.nslots = (int)std::min<long long>(ns, moe::kMaxSlots);
  p.q = std::max(1, std::min(moe::kNC, p.slot_bytes / p.pair_bytes));
  p.qr = std::max(1, std::min(moe::kNC / 2, p.slot_bytes / p.rpair_bytes));
  p.dq = (int)(p.slot_bytes / rowt);
  p.sk_lag = p.q;
  // the final reduction stages this CTA's block of every CTA's partial sums in the ring
  p.nrp = (int)round_up((size_t)(H + G - 1) / G, 4);
  if ((long long)G * maxm * p.nrp * 4 > (long long)p.nslots * p.slot_bytes || (long long)G * maxm * p.nrp * 4 >= (1 << 20))
    return MOE_ERR_UNSUPPORTED;
  p.nslots_x = p.nslots_d = p.hs_pairs = p.hs_perslot = 0;
  p.hs_nbuf = 1;
  p.d_rows_stage = p.dq;
  p.smem_bytes = p.off_ring + p.nslots * p.slot_bytes + 1024;
  return MOE_OK;
}

const void* kernel_for(const Params& p, int maxm_t, int phases) {
  return p.fmt == moe::FMT_BF16    ? moe::kernel_bf16(maxm_t, phases)
         : p.fmt == moe::FMT_NVFP4 ? moe::kernel_nvfp4(maxm_t, phases)
                                   : moe::kernel_fp8(maxm_t, phases);
}

moe_status check_weights(const moe_decode_config& c, const moe_decode_weights* w) {
  if (!w) return MOE_ERR_INVALID_ARG;
  auto need = [](const void* q) { return q != nullptr && aligned16(q); };
  if (!need(w->router_w) || !need(w->w13) || !need(w->w2)) return MOE_ERR_INVALID_ARG;
  if (c.score == MOE_SCORE_SIGMOID_BIAS && (!w->router_bias || (reinterpret_cast<uintptr_t>(w->router_bias) & 3u)))
    return MOE_ERR_INVALID_ARG;
  const bool fp4 = c.wdtype == MOE_W_NVFP4, fp8 = c.wdtype == MOE_W_FP8_BLOCK;
  if (fp4 && (!need(w->w13_scale) || !need(w->w2_scale) || !w->w13_gscale || !w->w2_gscale))
    return MOE_ERR_INVALID_ARG;
  if (fp8 && (!need(w->w13_scale) || !need(w->w2_scale))) return MOE_ERR_INVALID_ARG;
  if (c.num_shared > 0) {
    if (!need(w->sh_w13) || !need(w->sh_w2)) return MOE_ERR_INVALID_ARG;
    if (fp4 && (!need(w->sh_w13_scale) || !need(w->sh_w2_scale) || !w->sh_w13_gscale ||
                !w->sh_w2_gscale))
      return MOE_ERR_INVALID_ARG;
    if (fp8 && (!need(w->sh_w13_scale) || !need(w->sh_w2_scale))) return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Weight and scratch pointers of `from` into `to` (two layouts of one handle).
void bind_pointers(const Params& from, Params& to) {
  to.router_w = from.router_w;
  to.router_bias = from.router_bias;
  to.w13 = from.w13;
  to.w13_s = from.w13_s;
  to.w13_gs = from.w13_gs;
  to.w2 = from.w2;
  to.w2_s = from.w2_s;
  to.w2_gs = from.w2_gs;
  to.sh_w13 = from.sh_w13;
  to.sh_w13_s = from.sh_w13_s;
  to.sh_w13_gs = from.sh_w13_gs;
  to.sh_w2 = from.sh_w2;
  to.sh_w2_s = from.sh_w2_s;
  to.sh_w2_gs = from.sh_w2_gs;
  to.logits = from.logits;
  to.hbuf = from.hbuf;
  to.xflags = from.xflags;
  to.ctrl = from.ctrl;
  to.hist = from.hist;
  to.psum = from.psum;
}

// Whether a persistent run of m rows takes the expert-range kernel: always when
// forced (mode 2), else (mode 1) for one row.
bool use_flat(const moe_decode_handle* h, int m) {
  if (h->sk || h->sched != MOE_SCHED_PERSISTENT || !h->has_flat) return false;
  return h->flat_mode == 2 || (h->flat_mode == 1 && m == 1);
}
// Whether a persistent run of m rows takes the slot-interleaved kernel: always
// when forced (mode 2), else (mode 1) where it measured faster on GB300 -- one
// token row with bf16 weights (FP8 one-row: 41.1 us interleaved against 35.3
// phase-ordered).
bool interleaved(const moe_decode_handle* h, int m) {
  if (h->sk || h->sched != MOE_SCHED_PERSISTENT || !h->has_ilv || use_flat(h, m)) return false;
  return h->ilv_mode == 2 || (h->ilv_mode == 1 && h->base.fmt == moe::FMT_BF16 && m == 1);
}
// The layout a run of m rows uses.
const Params& active_params(const moe_decode_handle* h, int m) {
  return use_flat(h, m) ? h->flat : interleaved(h, m) ? h->ilv : h->base;
}
int threads_for(const moe_decode_handle* h, int m) {
  return use_flat(h, m) ? moe::kThreadsFlat : interleaved(h, m) ? moe::kThreadsIlv : moe::kThreads;
}

// The row bound of the kernel instantiation a launch of m rows takes: 1, 6
// (bf16 / FP8 phase-ordered and chained kernels: fewer registers for the
// per-row sums) or 8.
int maxm_for(const Params& p, int m, bool six_ok) {
  return m == 1 ? 1 : (m <= 6 && six_ok && p.fmt != moe::FMT_NVFP4) ? 6 : 8;
}

moe_status launch(moe_decode_handle* h, const Params& p, cudaStream_t stream) {
  const bool ilv = interleaved(h, p.M);
  const bool flat = use_flat(h, p.M);
  const int maxm_t = maxm_for(p, p.M, !h->sk && !ilv && !flat);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(threads_for(h, p.M));
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  void* args[] = {const_cast<Params*>(&p)};
  if (h->sched == MOE_SCHED_PERSISTENT) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.numAttrs = 1;
    const void* k = h->sk ? moe::kernel_sk(p.fmt, maxm_t)
                    : flat ? moe::kernel_flat(maxm_t)
                           : kernel_for(p, maxm_t, ilv ? moe::PH_ILV : moe::PH_ALL);
    if (cudaLaunchKernelExC(&cfg, k, args) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const int phases[3] = {moe::PH_R, moe::PH_U, moe::PH_D};
  for (int i = 0; i < 3; ++i) {
    cfg.numAttrs = 0;
    if (h->sched == MOE_SCHED_PDL_CHAIN) {
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.numAttrs = 1;
    }
    if (cudaLaunchKernelExC(&cfg, kernel_for(p, maxm_t, phases[i]), args) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace

namespace moe {
moe_status check_config_host(const moe_decode_config* cfg) { return check_config(cfg); }
moe_status check_weights_host(const moe_decode_config& cfg, const moe_decode_weights* w) {
  return check_weights(cfg, w);
}
moe_status plan_host(const moe_decode_config& cfg, int sms, int smem_optin, Params& p, bool ilv) {
  return plan(cfg, sms, smem_optin, p, ilv);
}
void bind_weights_host(const moe_decode_weights& w, Params& p) {
  p.router_w = static_cast<const uint8_t*>(w.router_w);
  p.router_bias = w.router_bias;
  p.w13 = static_cast<const uint8_t*>(w.w13);
  p.w2 = static_cast<const uint8_t*>(w.w2);
  p.w13_s = static_cast<const uint8_t*>(w.w13_scale);
  p.w2_s = static_cast<const uint8_t*>(w.w2_scale);
  p.w13_gs = w.w13_gscale;
  p.w2_gs = w.w2_gscale;
  p.sh_w13 = static_cast<const uint8_t*>(w.sh_w13);
  p.sh_w2 = static_cast<const uint8_t*>(w.sh_w2);
  p.sh_w13_s = static_cast<const uint8_t*>(w.sh_w13_scale);
  p.sh_w2_s = static_cast<const uint8_t*>(w.sh_w2_scale);
  p.sh_w13_gs = w.sh_w13_gscale;
  p.sh_w2_gs = w.sh_w2_gscale;
}
}  // namespace moe

extern "C" {

int32_t moe_decode_abi_version(void) { return MOE_DECODE_ABI_VERSION; }

const char* moe_decode_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_OOM: return "device allocation failed";
  }
  return "unknown status";
}

moe_status moe_decode_config_check(const moe_decode_config* cfg) { return check_config(cfg); }

moe_status moe_decode_plan(const moe_decode_config* cfg, int32_t sms, int32_t smem_optin, int32_t interleaved,
                           moe_decode_plan_info* out) {
  if (!out || sms <= 0 || smem_optin <= 0 || interleaved < 0 || interleaved > 2) return MOE_ERR_INVALID_ARG;
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  Params p;
  if (cfg->w2_layout == MOE_W2_I_H) {  // one layout: the split-K kernel's
    if (interleaved != 0) return MOE_ERR_UNSUPPORTED;
    st = plan_sk(*cfg, sms, smem_optin, p);
  } else {
    st = interleaved == 2 ? plan_flat(*cfg, sms, smem_optin, p) : plan(*cfg, sms, smem_optin, p, interleaved != 0);
  }
  if (st != MOE_OK) return st;
  out->smem_bytes = p.smem_bytes;
  out->ring_slots = p.nslots;
  out->slot_bytes = p.slot_bytes;
  out->extra_slots = p.nslots_x;
  out->down_slot_in_x = p.nslots_d;
  out->pairs_per_stage = p.q;
  out->router_pairs_per_stage = p.qr;
  out->down_rows_per_stage = p.d_rows_stage;
  out->h_pairs = p.hs_pairs;
  out->h_buffers = p.hs_nbuf;
  out->h_per_slot = p.hs_perslot;
  out->slots_max = p.nslot_max;
  out->pairs_max = p.npair_max;
  out->lag = interleaved == 1 ? p.ilv_lag : 0;
  out->down_h_offset = interleaved == 1 ? p.d_hoff : 0;
  out->threads = interleaved == 2 ? moe::kThreadsFlat : interleaved ? moe::kThreadsIlv : moe::kThreads;
  out->h_rows_max = p.sk_rows_max;
  out->down_t_rows_per_stage = p.dq;
  return MOE_OK;
}

moe_status moe_decode_create(const moe_decode_config* cfg, const moe_decode_weights* w,
                             moe_decode_handle** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  if ((st = check_weights(*cfg, w)) != MOE_OK) return st;
  int dev = 0, sms = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  Params p, pi;
  const bool sk = cfg->w2_layout == MOE_W2_I_H;
  if ((st = sk ? plan_sk(*cfg, sms, optin, p) : plan(*cfg, sms, optin, p, false)) != MOE_OK) return st;
  const bool has_ilv =
      !sk && kernel_for(p, 1, moe::PH_ILV) != nullptr && plan(*cfg, sms, optin, pi, true) == MOE_OK;
  Params pf;
  bool has_flat = !sk && plan_flat(*cfg, sms, optin, pf) == MOE_OK;
  // Every kernel this handle may launch gets the shared-memory size, and one
  // CTA of the single-kernel schedule must fit on every SM.
  const int phases[4] = {moe::PH_ALL, moe::PH_R, moe::PH_U, moe::PH_D};
  for (int mt : {1, 6, 8}) {
    if (mt == 6 && (sk || kernel_for(p, 6, moe::PH_ALL) == nullptr)) continue;  // bf16 / FP8 only
    if (sk) {
      const void* k = moe::kernel_sk(p.fmt, mt);
      int blocks = 0;
      if (!k) return MOE_ERR_UNSUPPORTED;
      if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k, moe::kThreads, p.smem_bytes) != cudaSuccess)
        return MOE_ERR_CUDA;
      if (blocks < 1) return MOE_ERR_UNSUPPORTED;
      continue;
    }
    for (int ph : phases) {
      const void* k = kernel_for(p, mt, ph);
      if (!k) return MOE_ERR_UNSUPPORTED;
      if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes) != cudaSuccess)
        return MOE_ERR_CUDA;
      int blocks = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k, moe::kThreads, p.smem_bytes) != cudaSuccess)
        return MOE_ERR_CUDA;
      if (blocks < 1) return MOE_ERR_UNSUPPORTED;
    }
    if (has_flat && mt != 6) {
      const void* k = moe::kernel_flat(mt);
      int blocks = 0;
      if (!k || cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, pf.smem_bytes) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k, moe::kThreadsFlat, pf.smem_bytes) != cudaSuccess)
        return MOE_ERR_CUDA;
      if (blocks < 1) has_flat = false;
    }
    if (has_ilv && mt != 6) {
      const void* k = kernel_for(pi, mt, moe::PH_ILV);
      int blocks = 0;
      if (!k || cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, pi.smem_bytes) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k, moe::kThreadsIlv, pi.smem_bytes) != cudaSuccess)
        return MOE_ERR_CUDA;
      if (blocks < 1) return MOE_ERR_UNSUPPORTED;
    }
  }
  // scratch: control words and the run_host outputs | logits | h | x flags | run_host inputs
  const size_t H = cfg->hidden, I = cfg->inter, E = cfg->num_experts, K = cfg->top_k;
  const size_t maxm = cfg->max_rows;
  // the control words (the status among them), then run_host's topk_idx, topk_w and
  // output rows: one device-to-host copy brings back a run's results and status
  const size_t o_ctrl = 0;
  const size_t o_si = round_up(moe::CTRL_WORDS * 4, 16);
  const size_t o_sw = o_si + round_up(maxm * K * 4, 16);
  const size_t o_so = o_sw + round_up(maxm * K * 4, 16);
  const size_t rb_bytes = o_so + maxm * H * 2;
  size_t off = round_up(rb_bytes, 256);
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, 256);
    return at;
  };
  const size_t o_logits = take(moe::kLogitRep * maxm * E * 8);
  const size_t o_h = take((size_t)moe::kHRep * p.npair_max * I * 4);
  const size_t o_xf = take((size_t)p.grid * 8);

  // expert-range kernel: tagged per-(block, slot, row) outputs
  const size_t o_y = has_flat ? take((size_t)p.grid * p.nslot_max * maxm * pf.flat_rb * 8) : 0;
  const size_t tag_end = off;
  // split-K kernel: every CTA's partial sums, by destination block
  const size_t o_ps = sk ? take((size_t)p.grid * p.grid * p.maxm * p.nrp * 4) : 0;
  // speculative expert prefetch: the predicted expert lists by run parity (-1: none)
  const size_t o_hist = take(2 * moe::kPfMax * 4);
  const size_t hist_end = off;
  const size_t o_sx = take(maxm * H * 2);
  const size_t o_sr = take(maxm * H * 2);
  auto* h = new (std::nothrow) moe_decode_handle();
  if (!h) return MOE_ERR_OOM;
  if (cudaMalloc(&h->scratch, off) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return MOE_ERR_OOM;
  }
  if (cudaHostAlloc(reinterpret_cast<void**>(&h->host_rb), rb_bytes, cudaHostAllocDefault) !=
      cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->scratch);
    delete h;
    return MOE_ERR_OOM;
  }
  uint8_t* base = static_cast<uint8_t*>(h->scratch);
  if (cudaMemset(base, 0, o_logits) != cudaSuccess ||
      cudaMemset(base + o_logits, 0xff, tag_end - o_logits) != cudaSuccess ||
      cudaMemset(base + o_hist, 0xff, hist_end - o_hist) != cudaSuccess ||

      cudaDeviceSynchronize() != cudaSuccess) {
    cudaFreeHost(h->host_rb);
    cudaFree(h->scratch);
    delete h;
    return MOE_ERR_CUDA;
  }
  h->cfg = *cfg;
  h->device = dev;
  h->sched = cfg->sched;
  h->scratch_bytes = off;
  p.router_w = static_cast<const uint8_t*>(w->router_w);
  p.router_bias = w->router_bias;
  p.w13 = static_cast<const uint8_t*>(w->w13);
  p.w2 = static_cast<const uint8_t*>(w->w2);
  p.w13_s = static_cast<const uint8_t*>(w->w13_scale);
  p.w2_s = static_cast<const uint8_t*>(w->w2_scale);
  p.w13_gs = w->w13_gscale;
  p.w2_gs = w->w2_gscale;
  p.sh_w13 = static_cast<const uint8_t*>(w->sh_w13);
  p.sh_w2 = static_cast<const uint8_t*>(w->sh_w2);
  p.sh_w13_s = static_cast<const uint8_t*>(w->sh_w13_scale);
  p.sh_w2_s = static_cast<const uint8_t*>(w->sh_w2_scale);
  p.sh_w13_gs = w->sh_w13_gscale;
  p.sh_w2_gs = w->sh_w2_gscale;
  p.ctrl = reinterpret_cast<uint32_t*>(base + o_ctrl);
  p.logits = reinterpret_cast<unsigned long long*>(base + o_logits);
  p.hbuf = reinterpret_cast<float*>(base + o_h);
  p.xflags = reinterpret_cast<unsigned long long*>(base + o_xf);
  if (sk) p.psum = reinterpret_cast<float*>(base + o_ps);
  p.hist = reinterpret_cast<int*>(base + o_hist);
  p.pf_n = 0;

  h->stage_x = reinterpret_cast<uint16_t*>(base + o_sx);
  h->stage_r = reinterpret_cast<uint16_t*>(base + o_sr);
  h->stage_out = reinterpret_cast<uint16_t*>(base + o_so);
  h->stage_idx = reinterpret_cast<int32_t*>(base + o_si);
  h->stage_w = reinterpret_cast<float*>(base + o_sw);
  h->rb_si = o_si;
  h->rb_sw = o_sw;
  h->rb_so = o_so;
  h->base = p;
  h->max_slots = p.nslots;
  h->has_ilv = has_ilv;
  h->has_flat = has_flat;
  h->sk = sk;
  h->max_slots_flat = has_flat ? pf.nslots : 0;
  if (has_flat) {
    bind_pointers(p, pf);
    pf.ybuf = reinterpret_cast<unsigned long long*>(base + o_y);
    h->flat = pf;
  }
  if (has_ilv) {
    // the interleaved layout, with the same weights and scratch
    bind_pointers(p, pi);
    h->ilv = pi;
    h->max_slots_ilv = pi.nslots;
  }
  *out = h;
  return MOE_OK;
}

moe_status moe_decode_run(moe_decode_handle* h, const void* x, const void* residual, void* out,
                          int32_t m_rows, int32_t* topk_idx, float* topk_w, moe_stream_t stream) {
  if (!h || !x || !residual || !out) return MOE_ERR_INVALID_ARG;
  if (m_rows < 1 || m_rows > h->cfg.max_rows) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(residual) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(topk_idx) & 3u) || (reinterpret_cast<uintptr_t>(topk_w) & 3u))
    return MOE_ERR_INVALID_ARG;
  // at most kMaxRowsLaunch rows per launch: a wider verify batch (up to
  // kMaxRowsRun rows) runs as row groups one after another on the stream, each a
  // complete layer step of its rows (rows are independent; the groups share the
  // handle's scratch in stream order)
  for (int g0 = 0; g0 < m_rows; g0 += moe::kMaxRowsLaunch) {
    const int mg = std::min(moe::kMaxRowsLaunch, m_rows - g0);
    Params p = active_params(h, mg);
    p.M = mg;
    const size_t row0 = (size_t)g0 * p.H;
    p.x = static_cast<const uint16_t*>(x) + row0;
    p.resid = static_cast<const uint16_t*>(residual) + row0;
    p.out = static_cast<uint16_t*>(out) + row0;
    p.topk_idx = topk_idx ? topk_idx + (size_t)g0 * p.K : nullptr;
    p.topk_w = topk_w ? topk_w + (size_t)g0 * p.K : nullptr;
    const size_t bytes = (size_t)mg * p.H * 2;
    p.out_aliases_x = overlaps(p.x, bytes, p.out, bytes) ? 1 : 0;
    const moe_status st = launch(h, p, reinterpret_cast<cudaStream_t>(stream));
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

moe_status moe_decode_get_status(moe_decode_handle* h, moe_stream_t stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t ctrl[4] = {0, 0, 0, 0};
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(ctrl, h->base.ctrl, sizeof(ctrl), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (ctrl[moe::CTRL_STATUS] == 0) return MOE_OK;
  if (cudaMemsetAsync(h->base.ctrl + moe::CTRL_STATUS, 0, 2 * sizeof(uint32_t), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_ERR_DEVICE_TIMEOUT;
}

moe_status moe_decode_run_host(moe_decode_handle* h, const void* x_host, const void* residual_host,
                               void* out_host, int32_t m_rows, int32_t* topk_idx_host,
                               float* topk_w_host, moe_stream_t stream) {
  if (!h || !x_host || !residual_host || !out_host) return MOE_ERR_INVALID_ARG;
  if (m_rows < 1 || m_rows > h->cfg.max_rows) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)m_rows * h->cfg.hidden * 2;
  const size_t kb = (size_t)m_rows * h->cfg.top_k * 4;
  // one copy per distinct input buffer: a residual that is x itself is not sent twice
  const bool same = residual_host == x_host;
  if (cudaMemcpyAsync(h->stage_x, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      (!same && cudaMemcpyAsync(h->stage_r, residual_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess))
    return MOE_ERR_CUDA;
  moe_status st = moe_decode_run(h, h->stage_x, same ? h->stage_x : h->stage_r, h->stage_out, m_rows,
                                 topk_idx_host ? h->stage_idx : nullptr,
                                 topk_w_host ? h->stage_w : nullptr, stream);
  if (st != MOE_OK) return st;
  // the status words, top-k outputs and output rows back as one contiguous block
  // (they follow each other after the control words), then one wait
  const size_t skip = moe::CTRL_STATUS * sizeof(uint32_t);
  const size_t end = h->rb_so + bytes;
  if (cudaMemcpyAsync(h->host_rb + skip, static_cast<uint8_t*>(h->scratch) + skip, end - skip, cudaMemcpyDeviceToHost,
                      s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  std::memcpy(out_host, h->host_rb + h->rb_so, bytes);
  if (topk_idx_host) std::memcpy(topk_idx_host, h->host_rb + h->rb_si, kb);
  if (topk_w_host) std::memcpy(topk_w_host, h->host_rb + h->rb_sw, kb);
  uint32_t status;
  std::memcpy(&status, h->host_rb + skip, sizeof(status));
  if (status == 0) return MOE_OK;
  if (cudaMemsetAsync(h->base.ctrl + moe::CTRL_STATUS, 0, 2 * sizeof(uint32_t), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_ERR_DEVICE_TIMEOUT;
}

moe_status moe_decode_set_option(moe_decode_handle* h, int32_t option, int64_t value) {
  if (!h) return MOE_ERR_INVALID_ARG;
  switch (option) {
    case MOE_OPT_SCHED:
      if (value < MOE_SCHED_PERSISTENT || value > MOE_SCHED_CHAIN) return MOE_ERR_INVALID_ARG;
      if (h->sk && value != MOE_SCHED_PERSISTENT) return MOE_ERR_UNSUPPORTED;  // one kernel for transposed down rows
      h->sched = (int)value;
      return MOE_OK;
    case MOE_OPT_WAIT_TIMEOUT_NS:
      if (value <= 0) return MOE_ERR_INVALID_ARG;
      h->base.timeout_ns = h->ilv.timeout_ns = h->flat.timeout_ns = (unsigned long long)value;
      return MOE_OK;
    case MOE_OPT_TEST_FLAGS:
      if (value < 0 || value > moe::TEST_SKIP_LOGITS) return MOE_ERR_INVALID_ARG;
      h->base.test_flags = h->ilv.test_flags = h->flat.test_flags = (int)value;
      return MOE_OK;
    case MOE_OPT_RING_SLOTS:
      if (value < 2 || value > std::max({h->max_slots, h->max_slots_ilv, h->max_slots_flat}))
        return MOE_ERR_INVALID_ARG;
      h->base.nslots = std::min((int)value, h->max_slots);
      h->ilv.nslots = std::min((int)value, h->max_slots_ilv);
      h->flat.nslots = std::max(3, std::min((int)value, h->max_slots_flat));
      return MOE_OK;
    case MOE_OPT_STAMPS:
      if (value & 7) return MOE_ERR_INVALID_ARG;
      h->base.stamps = h->ilv.stamps = h->flat.stamps =
          reinterpret_cast<unsigned long long*>(static_cast<uintptr_t>(value));
      return MOE_OK;
    case MOE_OPT_INTERLEAVE:
      if (value < 0 || value > 2) return MOE_ERR_INVALID_ARG;
      h->ilv_mode = (int)value;
      return MOE_OK;
    case MOE_OPT_FLAT:
      if (value < 0 || value > 2) return MOE_ERR_INVALID_ARG;
      h->flat_mode = (int)value;
      return MOE_OK;
    case MOE_OPT_PREFETCH_EXPERTS:
      if (value < 0 || value > moe::kPfMax) return MOE_ERR_INVALID_ARG;
      h->base.pf_n = h->ilv.pf_n = h->flat.pf_n = (int)value;
      return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status moe_decode_get_info(moe_decode_handle* h, int32_t what, int64_t* value) {
  if (!h || !value) return MOE_ERR_INVALID_ARG;
  if (what >= MOE_INFO_PREDICTED && what < MOE_INFO_PREDICTED + moe::kPfMax) {
    // the next run's prefetch list: its parity is the run tag the next run takes
    uint32_t ep = 0;
    int32_t e = -1;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&ep, h->base.ctrl + moe::CTRL_EPOCH, sizeof(ep), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(&e, h->base.hist + (size_t)(ep & 1u) * moe::kPfMax + (what - MOE_INFO_PREDICTED), sizeof(e),
                   cudaMemcpyDeviceToHost) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    *value = e;
    return MOE_OK;
  }
  switch (what) {
    case MOE_OPT_SCHED: *value = h->sched; return MOE_OK;
    case MOE_OPT_WAIT_TIMEOUT_NS: *value = (int64_t)h->base.timeout_ns; return MOE_OK;
    case MOE_OPT_TEST_FLAGS: *value = h->base.test_flags; return MOE_OK;
    case MOE_OPT_RING_SLOTS: *value = active_params(h, 1).nslots; return MOE_OK;
    case MOE_OPT_STAMPS: *value = (int64_t)reinterpret_cast<uintptr_t>(h->base.stamps); return MOE_OK;
    case MOE_OPT_INTERLEAVE: *value = h->has_ilv ? h->ilv_mode : 0; return MOE_OK;
    case MOE_OPT_FLAT: *value = h->has_flat ? h->flat_mode : 0; return MOE_OK;
    case MOE_INFO_SPLIT_K: *value = h->sk ? 1 : 0; return MOE_OK;
    case MOE_OPT_PREFETCH_EXPERTS: *value = h->base.pf_n; return MOE_OK;
    case MOE_INFO_FLAT_ROWS: {
      int64_t mask = 0;
      for (int m = 1; m <= h->cfg.max_rows; ++m)
        if (use_flat(h, std::min(m, moe::kMaxRowsLaunch))) mask |= int64_t(1) << (m - 1);
      *value = mask;
      return MOE_OK;
    }
    case MOE_INFO_GRID: *value = h->base.grid; return MOE_OK;
    case MOE_INFO_THREADS: *value = threads_for(h, 1); return MOE_OK;
    case MOE_INFO_SMEM: *value = active_params(h, 1).smem_bytes; return MOE_OK;
    case MOE_INFO_RING_SLOTS: *value = active_params(h, 1).nslots; return MOE_OK;
    case MOE_INFO_SLOT_BYTES: *value = active_params(h, 1).slot_bytes; return MOE_OK;
    case MOE_INFO_KERNELS_PER_RUN: *value = h->sched == MOE_SCHED_PERSISTENT ? 1 : 3; return MOE_OK;
    case MOE_INFO_SCRATCH_BYTES: *value = (int64_t)h->scratch_bytes; return MOE_OK;
    case MOE_INFO_INTERLEAVED_ROWS: {
      int64_t mask = 0;
      for (int m = 1; m <= h->cfg.max_rows; ++m)
        if (interleaved(h, std::min(m, moe::kMaxRowsLaunch))) mask |= int64_t(1) << (m - 1);
      *value = mask;
      return MOE_OK;
    }
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status moe_decode_destroy(moe_decode_handle* h) {
  if (!h) return MOE_OK;
  cudaError_t e = cudaFree(h->scratch);  // cudaFree waits for outstanding work
  const cudaError_t eh = h->host_rb ? cudaFreeHost(h->host_rb) : cudaSuccess;
  delete h;
  return e == cudaSuccess && eh == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
