// decode_noalloc.cu -- indexer_decode without a plan and without allocating.
//
// Some callers cannot create a plan, because creating one calls cudaMalloc:
// a custom-op hook inside a serving engine that only hands the op its input
// and output buffers and owns every byte of device memory itself, or a
// latency-critical loop that must never call cudaMalloc (it can synchronise
// the whole device and take milliseconds).  This entry point runs the same
// two decode kernels as indexer_decode, with their scratch (per-split top-15
// candidates, per-request split bookkeeping, a status word) carved out of a
// fixed array that lives in this library's device image: it is created when
// the library's module is loaded on a device and held until the process
// exits.
//
// Host code may only use the array's symbol as a handle: its device address
// is looked up with cudaGetSymbolAddress, once per device, by the first call
// made with that device current, and cached (with the device's SM count)
// for the life of the process.  Make that first call before any stream
// capture.  The cache does not survive cudaDeviceReset on that device: a
// process that resets a device must not call this entry point on it again.
//
// Every call uses the same array, so two calls whose kernels overlap on the
// GPU (different streams, or different host threads) corrupt each other's
// results: serialise them.  Nothing in the array has to start at zero: every
// word a call reads was written earlier by the same call, and a call whose
// wait ran out (a GPU that stopped making progress for 2 s) writes -1 rows
// rather than merging what the array held before.
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include <cuda_runtime.h>

#include "../../include/nvfp4_indexer.h"
#include "internal.h"

using namespace nvfp4idx;

constexpr size_t kNoAllocScratchBytes = 4u << 20;   // 4 MiB per device

// The scratch.  In host code this name is only a handle for
// cudaGetSymbolAddress, never an address a kernel may be given.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

struct DeviceSlot {
  bool ready = false;
  unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
  int num_sms = 0;
};
DeviceSlot g_slots[kMaxDevices];
std::mutex g_mu;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" int indexer_decode_noalloc(const uint8_t* q, const uint8_t* kv_pages, int num_blocks,
                                      const int32_t* page_table, int pt_stride, const int32_t* seq_lens,
                                      int num_reqs, int query_len, int num_heads, int32_t* out,
                                      int32_t* status, cudaStream_t stream) {
  auto ret = [](int code, const std::string& msg) {
    nvfp4idx::set_last_error_text(msg.c_str());
    return code;
  };
  nvfp4idx::set_last_error_text("");
  if (!q || !kv_pages || !page_table || !seq_lens || !out)
    return ret(IDX_EINVAL, "indexer_decode_noalloc: NULL array argument");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv_pages) |
       reinterpret_cast<uintptr_t>(out)) & 15u)
    return ret(IDX_EINVAL, "indexer_decode_noalloc: q, kv_pages and out must be 16-byte aligned");
  if (!(num_heads == 1 || num_heads == 2 || num_heads == 4 || num_heads == 8))
    return ret(IDX_EUNSUPPORTED, "indexer_decode_noalloc: num_heads must be 1, 2, 4 or 8");
  if (query_len < 1 || query_len > 8)
    return ret(IDX_EUNSUPPORTED, "indexer_decode_noalloc: query_len must be 1..8");
  if (num_reqs < 1 || num_reqs > kMaxDecodeReqs)
    return ret(IDX_EINVAL, "indexer_decode_noalloc: num_reqs must be 1..4096");
  if (num_blocks < 1 || pt_stride < 1 || pt_stride > (1 << 20))
    return ret(IDX_EINVAL, "indexer_decode_noalloc: bad num_blocks or pt_stride");

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return ret(IDX_ECUDA, std::string("indexer_decode_noalloc: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return ret(IDX_EINVAL, "indexer_decode_noalloc: device id out of range");
  DeviceSlot slot;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceSlot& s = g_slots[dev];
    if (!s.ready) {   // once per device, with that device current
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess)
        return ret(IDX_ECUDA, std::string("indexer_decode_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
      int sms = 0, major = 0, minor = 0;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
      if (e != cudaSuccess)
        return ret(IDX_ECUDA, std::string("indexer_decode_noalloc: device query: ") + cudaGetErrorString(e));
      if (major != 10 || minor != 3)
        return ret(IDX_EUNSUPPORTED, "indexer_decode_noalloc: device is sm_" + std::to_string(major) +
                                         std::to_string(minor) + ", the kernels are built for sm_103a");
      s.scratch = static_cast<unsigned char*>(ptr);
      s.num_sms = sms;
      s.ready = true;
    }
    slot = s;
  }

  // carve the scratch: status | request info | per-slot bad flags | candidates
  const int R = query_len * num_heads;
  const int grid = slot.num_sms;        // one decode CTA per SM, as indexer_decode
  // candidate slots: one per split unit (a CTA, or a warp for requests of up
  // to 8 rows) and per request
  const size_t slots = (size_t)decode_split_units(R, kPagesNvfp4, grid) + (size_t)num_reqs;
  const size_t off_status = 0;
  const size_t off_info = align256(off_status + sizeof(int32_t));
  const size_t off_bad = align256(off_info + (size_t)num_reqs * sizeof(int2));
  const size_t off_cand = align256(off_bad + slots * sizeof(int32_t));
  const size_t need = off_cand + slots * (size_t)R * kHistK * sizeof(float2);
  if (need > kNoAllocScratchBytes) {
    char buf[256];
    snprintf(buf, sizeof(buf),
             "indexer_decode_noalloc: %d requests x %d rows need %zu bytes of scratch, the fixed array "
             "holds %zu; use indexer_plan/indexer_decode or fewer requests per call",
             num_reqs, R, need, kNoAllocScratchBytes);
    return ret(IDX_ENOSPACE, buf);
  }

  DecodeParams p{};
  p.q = q;
  p.kv = kv_pages;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.scores_dbg = nullptr;
  p.status = status ? status : reinterpret_cast<int32_t*>(slot.scratch + off_status);
  p.req_info = reinterpret_cast<int2*>(slot.scratch + off_info);
  p.slot_bad = reinterpret_cast<int32_t*>(slot.scratch + off_bad);
  p.cand = reinterpret_cast<float2*>(slot.scratch + off_cand);
  p.num_blocks = num_blocks;
  p.pt_stride = pt_stride;
  p.num_reqs = num_reqs;
  p.qlen = query_len;
  p.H = num_heads;
  p.R = R;
  p.dbg_stride = 0;
  p.wait_ns = kWaitLimitNs;
  e = launch_decode(p, grid, stream);
  if (e != cudaSuccess)
    return ret(IDX_ECUDA, std::string("indexer_decode_noalloc: launch: ") + cudaGetErrorString(e));
  return IDX_OK;
}
