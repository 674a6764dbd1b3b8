// moe_decode_run_static: the layer step for callers that cannot allocate device
// memory. Its scratch lives in a fixed-size array of device memory defined
// below at file scope, so the call needs no handle and allocates nothing.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/moe_decode.h"
#include "internal.h"
#include "kernel_table.h"
#include "moe_params.h"

namespace {

// Control words, router logits, h rows and per-CTA flags of one call. Every GPU
// that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[MOE_DECODE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
constexpr size_t kCtrlBytes = 1024;  // moe::CTRL_WORDS 32-bit words, padded
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices];  // device address of g_static_scratch per device

static_assert(kCtrlBytes >= moe::CTRL_WORDS * 4, "control words exceed their area");

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// With the device current: the array's device address (the name
// g_static_scratch in host code is only a stand-in, not that address). The
// address is resolved on every call, which is cheap; the first call on a device,
// and any call that finds a new address (the module was reloaded, e.g. after a
// cudaDeviceReset, which also zeroes the array), sets the array up again: control
// words zeroed and every tagged word set to a tag no run ever uses (a blocking
// memset).
moe_status setup_device(int dev, unsigned char** out) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  if (g_scratch_ptr[dev] != p) {
    unsigned char* b = static_cast<unsigned char*>(p);
    if (cudaMemset(b, 0, kCtrlBytes) != cudaSuccess ||
        cudaMemset(b + kCtrlBytes, 0xff, MOE_DECODE_STATIC_SCRATCH_BYTES - kCtrlBytes) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
      cudaGetLastError();
      g_scratch_ptr[dev] = nullptr;
      return MOE_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = static_cast<unsigned char*>(p);
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status moe_decode_run_static(const moe_decode_config* cfg, const moe_decode_weights* w,
                                            const void* x, const void* residual, void* out, int32_t m_rows,
                                            int32_t* topk_idx, float* topk_w, moe_stream_t stream) {
  moe_status st = moe::check_config_host(cfg);
  if (st != MOE_OK) return st;
  // the split-K kernel's partial sums (grid x grid blocks) do not fit the static array
  if (cfg->w2_layout != MOE_W2_H_I) return MOE_ERR_UNSUPPORTED;
  if (!x || !residual || !out || m_rows < 1 || m_rows > cfg->max_rows) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(residual) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(topk_idx) & 3u) || (reinterpret_cast<uintptr_t>(topk_w) & 3u))
    return MOE_ERR_INVALID_ARG;
  int dev = 0, sms = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  moe::Params p;
  // the slot-interleaved kernel where it measured faster (bf16 weights, one token
  // row) and its layout fits, else the phase-ordered one
  const bool ilv = cfg->wdtype == MOE_W_BF16 && m_rows == 1 && moe::plan_host(*cfg, sms, optin, p, true) == MOE_OK;
  if (!ilv && (st = moe::plan_host(*cfg, sms, optin, p, false)) != MOE_OK) return st;
  // scratch layout inside the static array; larger configs are rejected
  const size_t maxm = p.maxm, E = cfg->num_experts, I = cfg->inter;
  const size_t o_logits = kCtrlBytes;
  const size_t o_h = o_logits + round256((size_t)moe::kLogitRep * maxm * E * 8);
  const size_t o_xf = o_h + round256((size_t)moe::kHRep * p.npair_max * I * 4);
  const size_t need = o_xf + round256((size_t)p.grid * 8);
  if (need > MOE_DECODE_STATIC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;
  if ((st = moe::check_weights_host(*cfg, w)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the call waits for its step and reads the status back, which a stream under
  // capture cannot do: refuse before any device work
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return MOE_ERR_INVALID_ARG;
  unsigned char* base = nullptr;
  if ((st = setup_device(dev, &base)) != MOE_OK) return st;

  moe::bind_weights_host(*w, p);
  p.ctrl = reinterpret_cast<uint32_t*>(base);
  p.logits = reinterpret_cast<unsigned long long*>(base + o_logits);
  p.hbuf = reinterpret_cast<float*>(base + o_h);
  p.xflags = reinterpret_cast<unsigned long long*>(base + o_xf);
  // the row bound of the instantiation: 1, 6 (bf16 / FP8 phase-ordered, runs of
  // up to 6 rows: fewer registers for the per-row sums) or 8
  const int maxm_t = m_rows == 1 ? 1 : (!ilv && m_rows <= 6 && p.fmt != moe::FMT_NVFP4) ? 6 : 8;
  const int which = ilv ? moe::PH_ILV : moe::PH_ALL;
  const void* kernel = p.fmt == moe::FMT_BF16    ? moe::kernel_bf16(maxm_t, which)
                       : p.fmt == moe::FMT_NVFP4 ? moe::kernel_nvfp4(maxm_t, which)
                                                 : moe::kernel_fp8(maxm_t, which);
  if (!kernel) return MOE_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  // one CTA of the cooperative launch must fit on every SM (registers and threads
  // as well as shared memory), as moe_decode_create checks
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, ilv ? moe::kThreadsIlv : moe::kThreads,
                                                    p.smem_bytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (blocks < 1) return MOE_ERR_UNSUPPORTED;
  // a status left by an earlier call must not stop this one
  if (cudaMemsetAsync(p.ctrl + moe::CTRL_STATUS, 0, 2 * sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(p.grid);
  lc.blockDim = dim3(ilv ? moe::kThreadsIlv : moe::kThreads);
  lc.dynamicSmemBytes = p.smem_bytes;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  // rows in groups of at most kMaxRowsLaunch, one launch each (as moe_decode_run)
  for (int g0 = 0; g0 < m_rows; g0 += moe::kMaxRowsLaunch) {
    const int mg = m_rows - g0 < moe::kMaxRowsLaunch ? m_rows - g0 : moe::kMaxRowsLaunch;
    moe::Params q = p;
    q.M = mg;
    const size_t row0 = (size_t)g0 * p.H;
    q.x = static_cast<const uint16_t*>(x) + row0;
    q.resid = static_cast<const uint16_t*>(residual) + row0;
    q.out = static_cast<uint16_t*>(out) + row0;
    q.topk_idx = topk_idx ? topk_idx + (size_t)g0 * p.K : nullptr;
    q.topk_w = topk_w ? topk_w + (size_t)g0 * p.K : nullptr;
    const size_t bytes = (size_t)mg * p.H * 2;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(q.x), oa = reinterpret_cast<uintptr_t>(q.out);
    q.out_aliases_x = (xa < oa + bytes && oa < xa + bytes) ? 1 : 0;
    void* args[] = {&q};
    if (cudaLaunchKernelExC(&lc, kernel, args) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
  }
  // wait for the step and report its device status (the status word lives in
  // the shared array too, so it is read and cleared here)
  uint32_t status = 0;
  if (cudaMemcpyAsync(&status, p.ctrl + moe::CTRL_STATUS, sizeof(status), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (status != 0) {
    if (cudaMemsetAsync(p.ctrl + moe::CTRL_STATUS, 0, 2 * sizeof(uint32_t), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_ERR_DEVICE_TIMEOUT;
  }
  return MOE_OK;
}
