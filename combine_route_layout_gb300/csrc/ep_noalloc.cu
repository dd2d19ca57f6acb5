// Routing layout without any caller-provided or library-allocated device
// memory beyond the caller's inputs and outputs.
//
// Some callers cannot call cudaMalloc: plugins and embedded engines whose
// host application has already reserved all device memory in its own pool
// (another allocation fails or fragments that pool), and code paths that
// must not enter a device allocator at all. For them this entry point runs
// the same routing-layout kernel as ep_dispatch, with its scratch (per-token
// destination masks, in-chunk ranks, per-chunk counts and offsets, the
// last-CTA ticket and the error bits) held in one file-scope static device
// array. Every GPU that loads the library keeps that array (about 2.3 MiB)
// until the process exits. All calls share it and it keeps the last call's
// contents; each call clears the counters that must start at zero. Calls
// that overlap on the GPU (different streams, or different host threads on
// one device) race on the array and must be serialised by the caller.
//
// This operation has no counterpart on the pages: it is the layout half of
// dispatch (MORI-EP User Guide, section 3) exposed on its own.
#include <cstring>
#include <mutex>
#include <string>

#include "ep_kernels.cuh"

namespace ep {
namespace {

constexpr int64_t kMaxTokens = EP_NOALLOC_MAX_TOKENS;
constexpr int64_t kMaxChunks = kMaxTokens / kChunk + EP_MAX_WORLD_SIZE;
constexpr size_t kHeader = 256;  // error bits + ticket
constexpr size_t kMaskOff = kHeader;
constexpr size_t kLocalOff = kMaskOff + kMaxTokens * sizeof(uint32_t);
constexpr size_t kCntOff = kLocalOff + kMaxTokens * EP_MAX_WORLD_SIZE;
constexpr size_t kOffOff = kCntOff + kMaxChunks * EP_MAX_WORLD_SIZE * sizeof(int32_t);
constexpr size_t kScratchBytes = kOffOff + kMaxChunks * EP_MAX_WORLD_SIZE * sizeof(int32_t);
static_assert(kScratchBytes == EP_NOALLOC_SCRATCH_BYTES, "header constant out of date");

static __device__ __align__(256) unsigned char g_layout_scratch[kScratchBytes];

// Device address of g_layout_scratch per device: looked up again on every
// call that is not being captured into a graph (a device reset or another
// context on the ordinal can move the array), and reused from here while a
// capture is in progress.
std::mutex g_mu;
void* g_scratch_addr[256] = {};

// slot_map[token][rank] and src_token_pos from the layout kernel's masks,
// in-chunk ranks and chunk offsets; one thread per (token, rank).
__global__ void slots_from_layout_kernel(LayoutParams p, int32_t* slot_map, int32_t* src_pos) {
  const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t g = q / p.R;
  const int r = (int)(q - g * p.R);
  if (g >= (int64_t)p.R * p.Tmax) return;
  const int s = (int)(g / p.Tmax), t = (int)(g - (int64_t)s * p.Tmax);
  if (t >= p.ntok[s]) return;
  const uint32_t m = p.mask[g];
  int slot = -1;
  if ((m >> r) & 1u) {
    const int c = s * p.cpr + t / kChunk;
    slot = p.chunk_off[(int64_t)c * p.R + r] + p.local8[g * p.R + r];
    src_pos[(int64_t)r * p.R * p.Tmax + slot] = s * (p.R * p.Tmax) + t;
  }
  slot_map[g * p.R + r] = slot;
}

}  // namespace
}  // namespace ep

namespace {
ep_status noalloc_fail(ep_status st, const std::string& msg) {
  return ep::record_error(st, msg.c_str());
}
}  // namespace

extern "C" ep_status ep_routing_layout_noalloc(int32_t world_size,
                                               int32_t max_num_inp_token_per_rank,
                                               int32_t num_experts_per_rank,
                                               int32_t num_experts_per_token,
                                               const int32_t* indices, const int32_t* num_tokens,
                                               int32_t* recv_num_token, int32_t* src_token_pos,
                                               int32_t* slot_map, int32_t* error_flags,
                                               void* stream) {
  using namespace ep;
  const int R = world_size, T = max_num_inp_token_per_rank;
  const int E_r = num_experts_per_rank, k = num_experts_per_token;
  if (R < 1 || R > EP_MAX_WORLD_SIZE)
    return noalloc_fail(EP_ERR_INVALID_ARG, "world_size outside [1, 32]");
  if (T < 1 || k < 1 || k > EP_MAX_TOPK || E_r < 1 || (int64_t)R * E_r > EP_MAX_EXPERTS)
    return noalloc_fail(EP_ERR_INVALID_ARG, "invalid token, top-k or expert count");
  if ((int64_t)R * T > kMaxTokens)
    return noalloc_fail(EP_ERR_INVALID_ARG,
                        "world_size * max_num_inp_token_per_rank = " +
                            std::to_string((int64_t)R * T) + " exceeds the static scratch limit " +
                            std::to_string(kMaxTokens) + " (EP_NOALLOC_MAX_TOKENS)");
  if (!indices || !num_tokens || !recv_num_token || !src_token_pos || !slot_map)
    return noalloc_fail(EP_ERR_INVALID_ARG, "NULL argument");
  for (int s = 0; s < R; ++s)
    if (num_tokens[s] < 0 || num_tokens[s] > T)
      return noalloc_fail(EP_ERR_INVALID_ARG, "num_tokens outside [0, max_num_inp_token_per_rank]");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 256)
    return noalloc_fail(EP_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(st, &cap);
  if (e != cudaSuccess)
    return noalloc_fail(EP_ERR_CUDA, std::string("cudaStreamIsCapturing: ") + cudaGetErrorString(e));
  unsigned char* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (cap == cudaStreamCaptureStatusNone || !g_scratch_addr[dev]) {
      // With this device current: the host-side name g_layout_scratch is not
      // a device address; ask the runtime for it (the first call on a device
      // also commits the array under lazy module loading).
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_layout_scratch);
      if (e == cudaSuccess) {
        g_scratch_addr[dev] = p;
      } else if (!g_scratch_addr[dev]) {
        return noalloc_fail(EP_ERR_CUDA,
                            std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
      } else {
        (void)cudaGetLastError();  // keep the address found by an earlier call
      }
    }
    base = static_cast<unsigned char*>(g_scratch_addr[dev]);
  }
  // error bits and the last-CTA ticket must start at zero
  e = cudaMemsetAsync(base, 0, kHeader, st);
  if (e != cudaSuccess)
    return noalloc_fail(EP_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));

  LayoutParams p;
  memset(&p, 0, sizeof(p));
  p.R = R; p.Tmax = T; p.k = k; p.E_r = E_r; p.E = R * E_r;
  p.cpr = (T + kChunk - 1) / kChunk;
  p.nchunks = R * p.cpr;
  for (int s = 0; s < R; ++s) p.ntok[s] = num_tokens[s];
  p.idx = indices;
  p.err = reinterpret_cast<int32_t*>(base);
  p.ticket = reinterpret_cast<unsigned int*>(base + 16);
  p.mask = reinterpret_cast<uint32_t*>(base + kMaskOff);
  p.local8 = base + kLocalOff;
  p.chunk_cnt = reinterpret_cast<int32_t*>(base + kCntOff);
  p.chunk_off = reinterpret_cast<int32_t*>(base + kOffOff);
  p.recv_num_token = recv_num_token;
  e = launch_layout_2d(p, st);
  if (e != cudaSuccess)
    return noalloc_fail(EP_ERR_CUDA, std::string("layout launch: ") + cudaGetErrorString(e));
  const int64_t n = (int64_t)R * T * R;
  slots_from_layout_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(p, slot_map,
                                                                       src_token_pos);
  e = cudaGetLastError();
  if (e != cudaSuccess)
    return noalloc_fail(EP_ERR_CUDA, std::string("slot launch: ") + cudaGetErrorString(e));
  if (error_flags) {
    e = cudaMemcpyAsync(error_flags, base, sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess)
      return noalloc_fail(EP_ERR_CUDA, std::string("cudaMemcpyAsync: ") + cudaGetErrorString(e));
  }
  return EP_OK;
}
