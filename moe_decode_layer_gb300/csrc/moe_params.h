// Launch parameters shared by the host planner and the device kernels.
#pragma once
#include <cstdint>

namespace moe {

constexpr int kNC = 12;                  // consumer warps per CTA
constexpr int kMaxRowsLaunch = 8;        // token rows one kernel launch handles
constexpr int kMaxRowsRun = 16;          // token rows one run handles (launches of <= 8 rows)
constexpr int kThreads = (kNC + 1) * 32; // + one producer warp
constexpr int kThreadsIlv = kThreads + 64;  // slot-interleaved kernel: + two hand-off warps
constexpr int kRpgMax = 5;               // down-projection rows per thread group per stage (at most; 4 groups x 5 rows hold the 17 rows of a Ling-shaped CTA block)
constexpr int kRpgFp4 = 3;               // NVFP4: its 32-element chunks leave more groups, so fewer rows each
__host__ __device__ constexpr int rows_per_group(int fmt) { return fmt == 1 ? kRpgFp4 : kRpgMax; }
constexpr int kMaxSlots = 64;            // ring slots (upper bound for the barrier arrays)
constexpr int kCplBf16 = 16;             // 16-byte x chunks per lane kept in registers (H <= 4096)
constexpr int kCplFp4 = 4;               // 32-element x chunks per lane for NVFP4 (H <= 4096)
constexpr int kCplFp8 = 8;               // 16-element x chunks per lane for FP8 (H <= 4096)
constexpr int kFp8Block = 128;           // FP8 weights: one fp32 scale per 128 x 128 block
constexpr int kFp8StagedScaleMax = 4096; // FP8: per-expert scale bytes staged with the weights at most
constexpr int kStageTarget = 32768;      // ring slot size aimed for (bytes)
constexpr int kMinSlots = 4;             // ring slots kept before shrinking the h staging area
constexpr int kLogitRep = 4;             // copies of the router logits (spreads the all-CTA read)
constexpr int kHRep = 4;                 // copies of the h rows (spreads the all-CTA read)
constexpr int kCandMax = 64;             // top-k candidates ranked in parallel per row
constexpr int kPfMax = 16;               // experts a run may prefetch into L2 from the previous run's routing
constexpr int kRouterCopy = 4096;        // bytes per bulk copy of router rows (more copies in flight)

enum WFmt : int { FMT_BF16 = 0, FMT_NVFP4 = 1, FMT_FP8 = 2 };

// Phases a kernel runs: router + shared gate/up (R), routed gate/up (U),
// down + combine + residual (D).
enum Phase : int { PH_R = 1, PH_U = 2, PH_D = 4, PH_ALL = 7 };
// Kernel selector (not a phase set): the single kernel with the slot-interleaved
// schedule -- each CTA computes a block of rows of every union slot's gate/up
// items, and the down stage of slot s follows the gate/up items of slot s + lag.
constexpr int PH_ILV = 8;
// Kernel selector: the expert-range single kernel (each CTA owns a contiguous
// range of (expert, gate/up row) items and of (expert, output block) down stages).
constexpr int PH_FLAT = 16;
// Kernel selector: the split-K single kernel (down matrices stored transposed;
// each CTA applies the down projection to the h rows it computed and the output
// is a fixed-order sum of every CTA's partial sums).
constexpr int PH_SK = 32;
constexpr int kThreadsFlat = kThreadsIlv;  // consumers, producer, publisher, fetcher
constexpr int kFlatSegs = 3;               // down segments per CTA: shared block + <= 2 routed slots
constexpr int kFlatMaxChunks = 128;        // 16-byte chunks of a down row (I <= 1024 bf16)
constexpr int kIlvRot = 37;  // per slot, the CTA -> row-block map rotates by this many CTAs
constexpr int kIlvCnt = 8;   // per-CTA arrival counters of the interleaved schedule (slot s uses s % 8)
// Interleaved-schedule words in shared memory (off_ucnt): the arrival counters,
// then the down stages issued and the producer's done flag.
enum IlvWord : int { ILV_DISSUED = kIlvCnt, ILV_PDONE = kIlvCnt + 1, ILV_WORDS = kIlvCnt + 4 };

// Control words at the start of the handle's scratch.
// CTRL_UCOUNT / CTRL_SCOUNT (64-bit, 8-byte aligned word index): CTAs whose gate-up
// results / shared experts' gate-up results of the current run are stored; reset by
// the last CTA. (Router logits need no count: readers poll their run tags.) Words
// 4 and 5 are unused.
enum Ctrl : int { CTRL_EPOCH = 0, CTRL_EXIT = 1, CTRL_STATUS = 2, CTRL_WHERE = 3,
                  CTRL_UCOUNT = 6, CTRL_SCOUNT = 8, CTRL_SLOTCNT = 16, CTRL_WORDS = 176 };
// CTRL_SLOTCNT + s: gate/up items of union slot s whose h is stored (all CTAs of
// the run; complete at I). Used when every pair's h fits the h area at once.
constexpr int kHSlotBar = 32;  // per-slot h mbarriers: full-barrier entries kHSlotBar + s (s < 32)
// Device status bits and the wait that gave up first.
enum DevErr : uint32_t { DEV_ERR_TIMEOUT = 1u };
enum WaitSite : uint32_t {
  SITE_RING_FULL = 1,
  SITE_RING_EMPTY = 2,
  SITE_LOGITS = 3,
  SITE_HIDDEN = 4,
  SITE_XFLAGS = 5,
  SITE_DRAIN = 6,
  SITE_FLAGS = 7
};
// Test flags.
enum TestFlag : int { TEST_SKIP_LOGITS = 1 };
// Per-CTA phase timestamps (%globaltimer, ns) when Params::stamps is set:
// stamps[cta * kStampSlots + event].
enum Stamp : int {
  ST_START = 0,       // kernel entry
  ST_X_LOADED = 1,    // x rows in shared memory (consumers)
  ST_R_DONE = 2,      // this CTA's router + shared gate/up stages consumed (warp 0 view)
  ST_ROUTED = 3,      // top-k and expert union ready
  ST_U_DONE = 4,      // routed gate/up stages consumed (warp 0 view)
  ST_D_FIRST = 5,     // first down stage's inputs staged
  ST_D_DONE = 6,      // outputs written
  ST_D_SUMMED = 19,   // down sums of the last row block complete (before the output reduction)
  ST_P_R_ISSUED = 8,  // producer: last router / shared stage issued
  ST_P_ROUTE = 9,     // producer: routing received
  ST_P_U_ISSUED = 10, // producer: last routed gate/up stage issued
  ST_P_D_ISSUED = 11, // producer: last down stage issued
  ST_LOGITS = 12,     // all router logits seen (routing warp 0)
  ST_TOPK = 13,       // top-k of row 0 done
  ST_U_FLAGS = 14,    // the gate/up-done count reached the grid size
  ST_RFLAG = 16,      // this CTA's router logits stored
  ST_U_DATA = 17,     // warp 0's first routed gate/up stage landed
  ST_D_HWAIT_NS = 7,     // (sum, thread 0) ns waiting for h batches in the down phase
  ST_D_MATH_NS = 20,     // (sum, thread 0) ns in the down-stage arithmetic
  ST_D_BAR_NS = 21,      // (sum, thread 0) ns at the down phase's per-batch barriers
  ST_D_WAIT_NS = 22,     // (sum, warp 0) ns down-phase warp 0 waited for its stages
  ST_CLOCK_MHZ = 23,  // (value) SM clock cycles per microsecond over the kernel
  kStampSlots = 24
};

// Shared-memory words kept in the misc block.
// MISC_XMAX + m: bf16 bits of the largest |x| of row m (NVFP4: sets the row's
// power-of-two scale into fp16's range).
enum Misc : int { MISC_EPOCH = 0, MISC_NROUTED = 1, MISC_ABORT = 2, MISC_ULO = 3, MISC_UHI = 4, MISC_ROUTED = 5,
                  MISC_WTOT = 8,
                  MISC_XMAX = 16, MISC_WORDS = 32 };

struct Params {
  // shapes
  int H, I, E, K, S, M, maxm, fmt;
  int score;         // 0: softmax -> top-k -> renormalise; 1: sigmoid + bias selection
  float routed_scale;
  float rms_eps;
  int pre_rmsnorm;
  // weights (device, borrowed)
  const uint8_t* router_w;
  const float* router_bias;  // [E] selection bias (score 1)
  const uint8_t* w13;
  const uint8_t* w13_s;
  const float* w13_gs;
  const uint8_t* w2;
  const uint8_t* w2_s;
  const float* w2_gs;
  const uint8_t* sh_w13;
  const uint8_t* sh_w13_s;
  const float* sh_w13_gs;
  const uint8_t* sh_w2;
  const uint8_t* sh_w2_s;
  const float* sh_w2_gs;
  // activations
  const uint16_t* x;
  const uint16_t* resid;
  uint16_t* out;
  int32_t* topk_idx;
  float* topk_w;
  // scratch (device, owned by the handle)
  unsigned long long* logits;  // [kLogitRep][maxm][E] tagged
  float* hbuf;                 // [kHRep][npair_max][I]: h of each (expert, row) pair, pair order
  unsigned long long* xflags;  // [grid] tagged: this CTA has read x
  uint32_t* ctrl;              // CTRL_WORDS
  int out_aliases_x;
  // planned layout
  int nchunk_h;      // code chunks per gate/up row (16 bytes; FP8: 16 codes)
  int row13, sc13;   // code / scale bytes per gate/up row
  int nchunk_i;      // code chunks per down row (16 bytes; FP8: 8 codes)
  int row2, sc2;     // code / scale bytes per down row
  int pair_bytes;    // one gate row + one up row (codes and scales)
  int sc13e;         // FP8: bytes of one expert's gate/up block scales, copied behind every gate/up
                     // stage of that expert (0: the consumers read them from global memory)
  int sc2e;          // FP8: bytes of one expert's down block scales, copied into every down stage
                     // at d_soff (0: read from global memory)
  int d_soff;        // byte offset of the staged FP8 down scales inside a down stage's ring slot
  int rpair_bytes;   // two router rows
  int q, qr;         // gate/up pairs per stage, router row pairs per stage (<= kNC)
  int slot_bytes, nslots;
  int d_rows_stage;  // down rows per stage
  int tg, ng;        // threads per down group, groups
  int grid;
  int nslot_max;     // S + min(E, maxm * K)
  int npair_max;     // S * maxm + maxm * K: (expert, row) pairs with an h row
  int hs_pairs;      // h rows (pairs) the down phase holds in shared memory
  int hs_nbuf;       // 1: one batch buffer of hs_pairs; 2: two of hs_pairs / 2 (next batch in flight)
  // shared-memory offsets from the aligned base
  int off_hbar;      // [2] mbarriers of the h batch buffers
  int item_base;     // cost of a routed gate/up item with N rows: item_base + N
  int nslots_x;      // extra ring slots for the routed gate/up stages, in the h area
  int off_xslot;     // first extra slot (slots nslots .. nslots + nslots_x - 1)
  int nslots_d;      // 1: in the down phase slot nslots lies in the x area (x is dead by then)
  int hs_perslot;    // 1: all pairs fit the h area; the single-kernel schedule fetches each slot's h
                     // as soon as that slot's items are done (per-slot counts and mbarriers)
  int off_xfree;     // mbarrier: the consumers are done with x (single-kernel schedule)
  int off_full, off_empty, off_xbar, off_slot_seq, off_x, off_hs, off_sel_e, off_sel_w;
  int off_emask, off_bitmap, off_slot_of, off_slot_e, off_slot_mask, off_slot_w, off_pair_base;
  int off_lg, off_cand, off_lmax, off_ccount, off_thr, off_wtmp, off_wpc;  // routing scratch (in the hs area)
  int off_pair_sr;   // [npair_max] (slot << 4 | row) of each (slot, row) pair
  // slot-interleaved schedule
  int ilv_lag;       // the down stage of slot s follows the gate/up items of slot s + ilv_lag
  int d_hoff;        // byte offset of the h rows inside a down stage's ring slot
  int off_ucnt;      // [ILV_WORDS]: consumer warps done with a slot's gate/up items (cumulative
                     // per counter), down stages issued, producer done
  int off_dslot;     // [nslot_max] ring slot of each slot's down stage (producer)
  int off_red, off_misc, off_ring;
  int off_bias;      // [E] fp32 selection bias (score 1)
  int smem_bytes;  // dynamic shared memory requested (includes alignment slack)
  unsigned long long timeout_ns;
  int test_flags;
  unsigned long long* stamps;  // optional [grid][kStampSlots]
  // expert-range kernel
  unsigned long long* ybuf;  // [grid][nslot_max][maxm][flat_rb] tagged: each union slot's down
                             // output of output block b (run tag << 32 | fp32 bits)
  int flat_rb;         // rows of the largest output block, rounded up to even
  int off_acnt;        // [nslot_max] consumer warps done with a slot's gate/up items
  // split-K down schedule (down matrices stored transposed, [I][H] per expert)
  int w2t;             // 1: w2 / sh_w2 (and FP8 scales) are [E][I][H] ([E][I/128][H/128])
  int dq;              // transposed down rows per down stage
  int sk_lag;          // a down stage follows the gate/up stages of its rows by this many rows
  int sk_rows_max;     // h rows one CTA may hold (checked on the device)
  int nrp;             // output rows per CTA block, padded to a multiple of 4
  int off_hsk;         // [sk_rows_max][maxm] fp32 h of this CTA's rows
  int off_htag;        // [sk_rows_max] 1 once the row's h is stored
  int off_psb;         // mbarrier: the partial-sum block of this CTA landed
  int off_psum;        // [nrp] x (parts) fp32 staging for the fixed-order reduction
  float* psum;         // [grid (destination)][grid (source)][M][nrp] fp32 partial sums
  // speculative expert prefetch
  int pf_n;            // experts to prefetch into L2 while routing runs (0: off)
  int* hist;           // [2][kPfMax] expert ids (-1: none) by run parity: run r reads list r & 1
                       // and writes the list for run r + 1
};

}  // namespace moe
