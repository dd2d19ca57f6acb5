// libep host library: the C ABI declared in include/ep.h.
//
// Validates the EpDispatchCombineConfig-style config (MORI-EP User Guide,
// section 2), carves the caller's workspace, keeps the dispatch/combine/reset
// state machine of section 3 (reset() must separate iterations unless
// combine is called with call_reset), and enqueues the kernels. No function
// here allocates device memory or blocks the host, except ep_sync.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "ep_convert.cuh"
#include "ep_kernels.cuh"

namespace {

thread_local std::string g_last_error;

ep_status fail(ep_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

ep_status cuda_fail(cudaError_t e, const char* what) {
  return fail(EP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

enum State { kReady = 0, kDispatched = 1, kCombined = 2 };


// EP_COMBINE_AUTO picks the bulk-copy combine from this many source tokens on.
constexpr int64_t kBulkMinTokens = 8192;

int dtype_size(int dt) {
  switch (dt) {
    case EP_DTYPE_BF16: return 2;
    case EP_DTYPE_FP32: return 4;
    case EP_DTYPE_FP8_E4M3: return 1;
    case EP_DTYPE_FP4_E2M1X2: return 1;   // two elements per byte (row bytes = H/2)
    default: return 0;
  }
}

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Sizes derived from a config.
struct Geometry {
  int R, H, k, E_r, E, Tmax;
  int64_t cap, pcap;
  int cpr, nchunks, cpr_recv, nchunks_recv;
  bool quant, std_moe, layout2d, registered_in;  // layouts reserved by the config
  int64_t combine_in_row_bytes;
  int64_t in_row_bytes, out_row_bytes;
  int scale_row_bytes;       // received scale row bytes (0 = none)
  int in_scale_row_bytes;    // pass-through input scale row bytes
};

// Workspace pointers (or offsets when base == nullptr).
struct Carve {
  int32_t* err;
  unsigned int* tickets;     // [4]
  uint32_t* mask;
  uint8_t* local8;
  int32_t* chunk_cnt2d;
  int32_t* chunk_off2d;
  int32_t* recv_num_token;
  int32_t* slot_map;
  int32_t* src_pos;
  uint8_t* recv_x;
  uint8_t* recv_scales;
  float* recv_w;
  int32_t* recv_idx;
  uint16_t* local16;
  int32_t* chunk_cnt_std;
  int32_t* chunk_off_std;
  int32_t* expert_count;
  int32_t* expert_offset;
  int32_t* rank_rows;
  int32_t* rank_base;
  int64_t* layout_range;
  int32_t* row_map;
  int32_t* packed_src_info;
  uint8_t* packed_x;
  uint8_t* packed_scales;
  uint16_t* conv_local16;
  int32_t* conv_recv_rows;   // [R][cap][k] packed row of each receive-row slot (conversions)
  int32_t* conv_chunk_cnt;
  int32_t* conv_chunk_off;
  uint8_t* reg_combine_in;   // registered combine input [R][cap][H] (zero-copy mode)
  size_t total;
};

template <typename T>
void take(uint8_t* base, size_t& off, T*& ptr, size_t bytes) {
  ptr = reinterpret_cast<T*>(base ? base + off : nullptr);
  off = align_up(off + bytes);
}

Carve carve(const Geometry& g, uint8_t* base) {
  Carve c{};
  size_t off = 0;
  const int64_t R = g.R, T = g.Tmax, k = g.k;
  take(base, off, c.err, 4 * sizeof(int32_t));
  take(base, off, c.tickets, 4 * sizeof(unsigned int));
  if (g.layout2d) {
    take(base, off, c.mask, R * T * 4);
    take(base, off, c.local8, R * T * R);
    take(base, off, c.chunk_cnt2d, (size_t)g.nchunks * R * 4);
    take(base, off, c.chunk_off2d, (size_t)g.nchunks * R * 4);
    take(base, off, c.recv_num_token, R * 4);
    take(base, off, c.slot_map, R * T * R * 4);
    take(base, off, c.src_pos, R * g.cap * 4);
    take(base, off, c.recv_x, R * g.cap * g.out_row_bytes);
    take(base, off, c.recv_scales, R * g.cap * g.scale_row_bytes);
    take(base, off, c.recv_w, R * g.cap * k * 4);
    take(base, off, c.recv_idx, R * g.cap * k * 4);
  }
  if (g.std_moe) {
    take(base, off, c.local16, R * T * k * 2);
    take(base, off, c.chunk_cnt_std, (size_t)g.nchunks * g.E * 4);
    take(base, off, c.chunk_off_std, (size_t)g.nchunks * g.E * 4);
    take(base, off, c.expert_count, (size_t)g.E * 4);
    take(base, off, c.expert_offset, (size_t)g.E * 4);
    take(base, off, c.rank_rows, R * 4);
    take(base, off, c.rank_base, R * 4);
    take(base, off, c.layout_range, (size_t)g.E * R * 8);
    take(base, off, c.row_map, R * T * k * 4);
    take(base, off, c.packed_src_info, g.pcap * 4);
    take(base, off, c.packed_x, g.pcap * g.out_row_bytes);
    take(base, off, c.packed_scales, g.pcap * g.scale_row_bytes);
  }
  if (g.std_moe && g.layout2d) {  // the conversions between the two layouts
    take(base, off, c.conv_local16, R * g.cap * k * 2);
    take(base, off, c.conv_recv_rows, R * g.cap * k * 4);
    take(base, off, c.conv_chunk_cnt, (size_t)g.nchunks_recv * g.E_r * 4);
    take(base, off, c.conv_chunk_off, (size_t)g.nchunks_recv * g.E_r * 4);
  }
  if (g.registered_in) take(base, off, c.reg_combine_in, R * g.cap * g.combine_in_row_bytes);
  c.total = off;
  return c;
}

ep_status make_geometry(const ep_config* cfg, Geometry* g) {
  if (!cfg) return fail(EP_ERR_INVALID_ARG, "config is NULL");
  const int R = cfg->world_size, H = cfg->hidden_dim, k = cfg->num_experts_per_token;
  const int E_r = cfg->num_experts_per_rank, T = cfg->max_num_inp_token_per_rank;
  if (R < 1 || R > EP_MAX_WORLD_SIZE)
    return fail(EP_ERR_INVALID_ARG, "world_size %d outside [1, %d]", R, EP_MAX_WORLD_SIZE);
  if (H < 8 || H % 8 != 0) return fail(EP_ERR_INVALID_ARG, "hidden_dim %d must be a positive multiple of 8", H);
  if (k < 1 || k > EP_MAX_TOPK)
    return fail(EP_ERR_INVALID_ARG, "num_experts_per_token %d outside [1, %d]", k, EP_MAX_TOPK);
  if (E_r < 1 || (int64_t)R * E_r > EP_MAX_EXPERTS)
    return fail(EP_ERR_INVALID_ARG, "world_size * num_experts_per_rank must be in [1, %d]",
                EP_MAX_EXPERTS);
  if (T < 1) return fail(EP_ERR_INVALID_ARG, "max_num_inp_token_per_rank must be >= 1");
  if ((int64_t)R * R * T > INT32_MAX)
    return fail(EP_ERR_INVALID_ARG, "world_size^2 * max tokens exceeds the int32 src_token_pos range");
  const int in_sz = dtype_size(cfg->data_type);
  if (in_sz == 0) return fail(EP_ERR_INVALID_ARG, "unknown data_type %d", cfg->data_type);
  if (cfg->quant_type != EP_QUANT_NONE && cfg->quant_type != EP_QUANT_FP8_E4M3_BLOCK128 &&
      cfg->quant_type != EP_QUANT_FP4_E2M1_BLOCK32)
    return fail(EP_ERR_INVALID_ARG, "unknown quant_type %d", cfg->quant_type);
  const bool quant = cfg->quant_type != EP_QUANT_NONE;
  const int qblock = cfg->quant_type == EP_QUANT_FP4_E2M1_BLOCK32 ? 32 : EP_QUANT_BLOCK;
  if (cfg->combine_dtype != EP_DTYPE_BF16 && cfg->combine_dtype != EP_DTYPE_FP32)
    return fail(EP_ERR_INVALID_ARG, "combine_dtype must be BF16 or FP32");
  if (cfg->combine_out_dtype != EP_DTYPE_BF16 && cfg->combine_out_dtype != EP_DTYPE_FP32)
    return fail(EP_ERR_INVALID_ARG, "combine_out_dtype must be BF16 or FP32");
  if (cfg->scale_dim < 0) return fail(EP_ERR_INVALID_ARG, "scale_dim must be >= 0");
  if (cfg->scale_dim > 0 && cfg->scale_type_size != 1 && cfg->scale_type_size != 2 &&
      cfg->scale_type_size != 4 && cfg->scale_type_size != 8)
    return fail(EP_ERR_INVALID_ARG, "scale_type_size must be 1, 2, 4 or 8");
  if (cfg->warp_num_per_block > 8)
    return fail(EP_ERR_INVALID_ARG, "warp_num_per_block must be <= 8");
  if (cfg->combine_impl < EP_COMBINE_AUTO || cfg->combine_impl > EP_COMBINE_BULK)
    return fail(EP_ERR_INVALID_ARG, "unknown combine_impl %d", cfg->combine_impl);
  if (cfg->dispatch_impl < EP_DISPATCH_AUTO || cfg->dispatch_impl > EP_DISPATCH_BULK)
    return fail(EP_ERR_INVALID_ARG, "unknown dispatch_impl %d", cfg->dispatch_impl);
  Geometry x{};
  x.R = R; x.H = H; x.k = k; x.E_r = E_r; x.E = R * E_r; x.Tmax = T;
  x.cap = (int64_t)R * T;
  x.cpr = (T + ep::kChunk - 1) / ep::kChunk;
  x.nchunks = R * x.cpr;
  x.cpr_recv = (int)((x.cap + ep::kChunk - 1) / ep::kChunk);
  x.nchunks_recv = R * x.cpr_recv;
  x.quant = quant;
  if (cfg->standard_moe < 0 || cfg->standard_moe > 2)
    return fail(EP_ERR_INVALID_ARG, "standard_moe must be 0 (2D layout), 1 (packed layout) or 2 (both)");
  x.std_moe = cfg->standard_moe != 0;
  x.layout2d = cfg->standard_moe != 1;
  x.registered_in = cfg->use_external_inp_buf == 0;
  if (x.registered_in && !x.layout2d)
    return fail(EP_ERR_INVALID_ARG, "use_external_inp_buf = 0 needs the 2D layout (standard_moe 0 or 2)");
  x.combine_in_row_bytes = (int64_t)H * dtype_size(cfg->combine_dtype);
  x.in_row_bytes = cfg->data_type == EP_DTYPE_FP4_E2M1X2 ? (int64_t)H / 2 : (int64_t)H * in_sz;
  if (cfg->data_type == EP_DTYPE_FP4_E2M1X2 && H % 32 != 0)
    return fail(EP_ERR_INVALID_ARG, "packed FP4 input needs hidden_dim %% 32 == 0");
  if (x.in_row_bytes % 16 != 0)
    return fail(EP_ERR_INVALID_ARG, "hidden_dim * element size must be a multiple of 16 bytes");
  if (quant) {
    if (cfg->data_type != EP_DTYPE_BF16)
      return fail(EP_ERR_INVALID_ARG, "block quantisation needs BF16 input");
    if (H % qblock != 0)
      return fail(EP_ERR_INVALID_ARG, "block quantisation needs hidden_dim %% %d == 0", qblock);
    if (cfg->scale_dim != 0 && !(cfg->scale_dim == H / qblock && cfg->scale_type_size == 4))
      return fail(EP_ERR_INVALID_ARG,
                  "with block quantisation scale_dim must be 0 or hidden_dim/%d (4-byte)", qblock);
    x.out_row_bytes = cfg->quant_type == EP_QUANT_FP4_E2M1_BLOCK32 ? H / 2 : H;
    x.scale_row_bytes = H / qblock * 4;
    x.in_scale_row_bytes = 0;
  } else {
    x.out_row_bytes = x.in_row_bytes;
    x.scale_row_bytes = cfg->scale_dim * (cfg->scale_dim > 0 ? cfg->scale_type_size : 0);
    x.in_scale_row_bytes = x.scale_row_bytes;
  }
  if (x.std_moe) {
    // one pool for all ranks: at most one row per (token, slot), plus at most
    // 127 padding rows per expert, whatever the routing
    const int64_t worst = (int64_t)R * T * k + (int64_t)(ep::kPadRows - 1) * R * E_r;
    x.pcap = cfg->max_packed_rows_per_rank > 0 ? (int64_t)R * cfg->max_packed_rows_per_rank : worst;
    if (x.pcap > INT32_MAX)
      return fail(EP_ERR_INVALID_ARG, "packed pool rows exceed int32");
  } else {
    x.pcap = 0;
  }
  *g = x;
  return EP_OK;
}

ep_status device_sm_count(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  *out = n;
  return EP_OK;
}

}  // namespace

int ep::ctas_per_sm(const void* kernel, int block, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, size_t, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  const auto key = std::make_tuple(kernel, block, smem, dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  if (smem > 48 * 1024) {
    // the limit is a property of the kernel, not of one launch: raise it to the
    // device maximum (less the kernel's static shared memory) so launches of
    // other sizes keep working
    int optin = 0;
    cudaFuncAttributes fa{};
    if (dev < 0 ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, kernel) != cudaSuccess)
      optin = 0;
    const int most = optin - (int)fa.sharedSizeBytes;
    (void)cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               most > (int)smem ? most : (int)smem);
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, block, smem) != cudaSuccess ||
      n < 1)
    n = 1;
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = n;
  return n;
}

ep_status ep::record_error(ep_status st, const char* msg) {
  g_last_error = msg;
  return st;
}

struct ep_handle {
  ep_config cfg;
  Geometry g;
  Carve w;
  uint8_t* ws;
  size_t ws_bytes;
  int state;
  bool has2d, hasstd, needs_init;
  int ntok[EP_MAX_WORLD_SIZE];
  int sm_count;
  int lc_blocks[2], lc_warps[2];  // launch configuration per ep_phase
};

namespace {

ep_status ensure_ready_device(ep_handle* h, cudaStream_t st) {
  if (h->sm_count == 0) {
    ep_status s = device_sm_count(&h->sm_count);
    if (s != EP_OK) return s;
  }
  if (h->needs_init) {
    cudaError_t e = cudaMemsetAsync(h->w.err, 0, 4 * sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->w.tickets, 0, 4 * sizeof(unsigned int), st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    h->needs_init = false;
  }
  return EP_OK;
}

// Launch configuration of a phase (EP_PHASE_DISPATCH: layout, dispatch and
// convert_dispatch_output; EP_PHASE_COMBINE: combine and convert_combine_input).
ep::LaunchCfg launch_cfg(const ep_handle* h, int phase) {
  ep::LaunchCfg lc;
  lc.grid_hint = h->lc_blocks[phase];
  lc.block = (h->lc_warps[phase] > 0 ? h->lc_warps[phase] : 8) * 32;
  lc.sm_count = h->sm_count;
  return lc;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Bulk-copy combine when asked for, or under EP_COMBINE_AUTO when it measured
// faster on GB300: the 2D layout with at least kBulkMinTokens source tokens
// (its four-stage ring needs several tokens per CTA to stay full; with fewer,
// and for the packed layout, the vector kernel was as fast or faster).
bool use_bulk(const ep_handle* h, const ep::CombineParams& p, bool std_layout) {
  if (h->cfg.combine_impl == EP_COMBINE_VECTOR) return false;
  if (!ep::combine_bulk_supported(p, std_layout)) return false;
  if (h->cfg.combine_impl == EP_COMBINE_BULK) return true;
  int64_t tokens = 0;
  for (int r = 0; r < h->g.R; ++r) tokens += h->ntok[r];
  return !std_layout && tokens >= kBulkMinTokens;
}

// Bulk-copy dispatch (copy mode only) when asked for, or under
// EP_DISPATCH_AUTO from kBulkMinTokens source tokens on (measured slightly
// faster there on GB300, slower for a handful of tokens).
bool use_bulk_dispatch(const ep_handle* h, const ep::DispatchParams& p) {
  if (h->g.quant || h->cfg.dispatch_impl == EP_DISPATCH_VECTOR) return false;
  if (!ep::dispatch_bulk_supported(p)) return false;
  if (h->cfg.dispatch_impl == EP_DISPATCH_BULK) return true;
  int64_t tokens = 0;
  for (int r = 0; r < h->g.R; ++r) tokens += h->ntok[r];
  return tokens >= kBulkMinTokens;
}

ep_status check_tokens(ep_handle* h, const int32_t* num_tokens) {
  if (!num_tokens) return fail(EP_ERR_INVALID_ARG, "num_tokens is NULL");
  for (int s = 0; s < h->g.R; ++s)
    if (num_tokens[s] < 0 || num_tokens[s] > h->g.Tmax)
      return fail(EP_ERR_INVALID_ARG, "num_tokens[%d] = %d outside [0, %d]", s, num_tokens[s],
                  h->g.Tmax);
  return EP_OK;
}

ep_status check_dispatch_inputs(ep_handle* h, const void* x, const float* w, const void* scales,
                                const int32_t* idx) {
  if (!x || !w || !idx) return fail(EP_ERR_INVALID_ARG, "x, weights and indices must be non-NULL");
  if (!aligned(x, 16)) return fail(EP_ERR_INVALID_ARG, "x must be 16-byte aligned");
  if (!aligned(w, 4) || !aligned(idx, 4))
    return fail(EP_ERR_INVALID_ARG, "weights and indices must be 4-byte aligned");
  if (h->g.quant && scales)
    return fail(EP_ERR_INVALID_ARG, "scales must be NULL with block quantisation (computed)");
  if (!h->g.quant && h->g.in_scale_row_bytes > 0 && !scales)
    return fail(EP_ERR_INVALID_ARG, "scale_dim > 0 needs a scales array");
  if (scales && (h->g.in_scale_row_bytes % 4 == 0) && !aligned(scales, 4))
    return fail(EP_ERR_INVALID_ARG, "scales must be 4-byte aligned");
  return EP_OK;
}

void fill_layout_common(ep_handle* h, const int32_t* idx, ep::LayoutParams* p) {
  const Geometry& g = h->g;
  memset(p, 0, sizeof(*p));
  p->R = g.R; p->Tmax = g.Tmax; p->k = g.k; p->E_r = g.E_r; p->E = g.E;
  p->cpr = g.cpr; p->nchunks = g.nchunks;
  for (int s = 0; s < g.R; ++s) p->ntok[s] = h->ntok[s];
  p->idx = idx;
  p->err = h->w.err;
}

void fill_dispatch_common(ep_handle* h, const void* x, const float* w, const void* scales,
                          const int32_t* idx, ep::DispatchParams* p) {
  const Geometry& g = h->g;
  memset(p, 0, sizeof(*p));
  p->R = g.R; p->Tmax = g.Tmax; p->k = g.k; p->E_r = g.E_r; p->E = g.E; p->cpr = g.cpr;
  for (int s = 0; s < g.R; ++s) p->ntok[s] = h->ntok[s];
  p->H = g.H;
  p->in_row_bytes = g.in_row_bytes;
  p->out_row_bytes = g.out_row_bytes;
  p->scale_row_bytes = g.quant ? 0 : g.in_scale_row_bytes;
  const int64_t step = g.quant ? (int64_t)ep::kQuantUnroll * 512 * 2
                               : (int64_t)ep::kCopyUnroll * 512;  // source bytes per unit
  p->segs_per_token = (int)((g.in_row_bytes + step - 1) / step);
  p->total_units = (int64_t)g.R * g.Tmax * p->segs_per_token;
  p->x = static_cast<const uint8_t*>(x);
  p->w = w;
  p->idx = idx;
  p->scales_in = static_cast<const uint8_t*>(scales);
}

}  // namespace

extern "C" {

const char* ep_last_error(void) { return g_last_error.c_str(); }

size_t ep_workspace_size(const ep_config* cfg) {
  Geometry g;
  if (make_geometry(cfg, &g) != EP_OK) return 0;
  return carve(g, nullptr).total;
}

ep_status ep_config_create(const ep_config* cfg, void* d_workspace, size_t workspace_bytes,
                           ep_handle** out_handle) {
  if (!out_handle) return fail(EP_ERR_INVALID_ARG, "out_handle is NULL");
  *out_handle = nullptr;
  Geometry g;
  ep_status s = make_geometry(cfg, &g);
  if (s != EP_OK) return s;
  const size_t need = carve(g, nullptr).total;
  if (!d_workspace) return fail(EP_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(d_workspace, kAlign)) return fail(EP_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (workspace_bytes < need)
    return fail(EP_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  ep_handle* h = new ep_handle();
  h->cfg = *cfg;
  for (int ph = 0; ph < 2; ++ph) {
    h->lc_blocks[ph] = cfg->block_num;
    h->lc_warps[ph] = cfg->warp_num_per_block;
  }
  h->g = g;
  h->ws = static_cast<uint8_t*>(d_workspace);
  h->ws_bytes = workspace_bytes;
  h->w = carve(g, h->ws);
  h->state = kReady;
  h->has2d = h->hasstd = false;
  h->needs_init = true;
  h->sm_count = 0;
  *out_handle = h;
  return EP_OK;
}

void ep_destroy(ep_handle* h) { delete h; }

ep_status ep_dispatch(ep_handle* h, const void* x, const float* weights, const void* scales,
                      const int32_t* indices, const int32_t* num_tokens, void* stream,
                      ep_dispatch_out* out) {
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  if (!h->g.layout2d)
    return fail(EP_ERR_INVALID_ARG,
                "standard_moe = 1 reserves only the packed layout (2 reserves both layouts)");
  if (h->state != kReady) return fail(EP_ERR_STATE, "dispatch needs reset() after the previous iteration");
  ep_status s = check_dispatch_inputs(h, x, weights, scales, indices);
  if (s == EP_OK) s = check_tokens(h, num_tokens);
  if (s != EP_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  s = ensure_ready_device(h, st);
  if (s != EP_OK) return s;
  for (int r = 0; r < h->g.R; ++r) h->ntok[r] = num_tokens[r];

  ep::LayoutParams lp;
  fill_layout_common(h, indices, &lp);
  lp.mask = h->w.mask;
  lp.local8 = h->w.local8;
  lp.recv_num_token = h->w.recv_num_token;
  lp.chunk_cnt = h->w.chunk_cnt2d;
  lp.chunk_off = h->w.chunk_off2d;
  lp.ticket = h->w.tickets + 0;

  ep::DispatchParams dp;
  fill_dispatch_common(h, x, weights, scales, indices, &dp);
  dp.cap = h->g.cap;
  dp.mask = h->w.mask;
  dp.local8 = h->w.local8;
  dp.chunk_off = h->w.chunk_off2d;
  dp.slot_map = h->w.slot_map;
  dp.src_pos = h->w.src_pos;
  dp.out_x = h->w.recv_x;
  dp.out_scales = h->w.recv_scales;
  dp.out_w = h->w.recv_w;
  dp.out_idx = h->w.recv_idx;
  dp.err = h->w.err;
  const bool bulk = use_bulk_dispatch(h, dp);
  if (!bulk && h->g.nchunks <= ep::kSmallScanChunks) {
    // small batch: the vector dispatch kernel sums the (few) chunk counts
    // itself, which takes the layout's last-CTA scan off the critical path
    lp.no_scan = 1;
    dp.chunk_cnt = h->w.chunk_cnt2d;
    dp.recv_num_token = h->w.recv_num_token;
  }
  cudaError_t e = ep::launch_layout_2d(lp, st);
  if (e != cudaSuccess) return cuda_fail(e, "routing-layout launch");
  e = bulk ? ep::launch_dispatch_bulk_copy(dp, false, launch_cfg(h, EP_PHASE_DISPATCH), st)
           : ep::launch_dispatch_2d(dp, h->g.quant ? h->cfg.quant_type : 0,
                                    launch_cfg(h, EP_PHASE_DISPATCH), st);
  if (e != cudaSuccess) return cuda_fail(e, "dispatch launch");

  h->state = kDispatched;
  h->has2d = true;
  h->hasstd = false;
  if (out) {
    out->x = h->w.recv_x;
    out->scales = h->g.scale_row_bytes > 0 ? h->w.recv_scales : nullptr;
    out->weights = h->w.recv_w;
    out->indices = h->w.recv_idx;
    out->recv_num_token = h->w.recv_num_token;
    out->src_token_pos = h->w.src_pos;
    out->cap = h->g.cap;
    out->x_row_bytes = h->g.out_row_bytes;
    out->scale_row_bytes = h->g.scale_row_bytes;
  }
  return EP_OK;
}

ep_status ep_combine(ep_handle* h, const void* expert_out, const float* weights,
                     const int32_t* indices, void* out, float* out_weights, int32_t call_reset,
                     void* stream) {
  (void)indices;
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  if (!h->has2d || h->state == kReady) return fail(EP_ERR_STATE, "combine needs a preceding dispatch");
  if (!expert_out) expert_out = h->w.reg_combine_in;  // zero-copy mode
  if (!expert_out || !out)
    return fail(EP_ERR_INVALID_ARG,
                "out must be non-NULL, and expert_out too unless use_external_inp_buf = 0");
  if (!aligned(expert_out, 16) || !aligned(out, 16))
    return fail(EP_ERR_INVALID_ARG, "expert_out and out must be 16-byte aligned");
  if ((h->cfg.weighted_combine || out_weights) && !weights)
    return fail(EP_ERR_INVALID_ARG, "weighted combine and out_weights need weights");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ep_status s = ensure_ready_device(h, st);
  if (s != EP_OK) return s;
  const Geometry& g = h->g;
  ep::CombineParams p;
  memset(&p, 0, sizeof(p));
  p.R = g.R; p.Tmax = g.Tmax; p.k = g.k; p.E_r = g.E_r; p.H = g.H;
  for (int r = 0; r < g.R; ++r) p.ntok[r] = h->ntok[r];
  p.cap = g.cap;
  p.segs_per_token = (g.H + ep::kCombineUnroll * 256 - 1) / (ep::kCombineUnroll * 256);
  p.total_units = (int64_t)g.R * g.Tmax * p.segs_per_token;
  p.weighted = h->cfg.weighted_combine != 0;
  p.y = static_cast<const uint8_t*>(expert_out);
  p.w = weights;
  p.recv_idx = h->w.recv_idx;
  p.slot_map = h->w.slot_map;
  p.out = static_cast<uint8_t*>(out);
  p.out_w = out_weights;
  p.err = h->w.err;
  cudaError_t e = use_bulk(h, p, false)
                      ? ep::launch_combine_2d_bulk(p, h->cfg.combine_dtype,
                                                   h->cfg.combine_out_dtype, launch_cfg(h, EP_PHASE_COMBINE), st)
                      : ep::launch_combine_2d(p, h->cfg.combine_dtype, h->cfg.combine_out_dtype,
                                              launch_cfg(h, EP_PHASE_COMBINE), st);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  h->state = kCombined;
  if (call_reset) return ep_reset(h, stream);
  return EP_OK;
}

ep_status ep_get_registered_combine_input_buffer(ep_handle* h, void** d_buffer) {
  if (!h || !d_buffer) return fail(EP_ERR_INVALID_ARG, "NULL argument");
  if (!h->w.reg_combine_in)
    return fail(EP_ERR_STATE, "config has use_external_inp_buf != 0: no registered buffer");
  *d_buffer = h->w.reg_combine_in;
  return EP_OK;
}

ep_status ep_get_dispatch_src_token_pos(ep_handle* h, const int32_t** d_src_token_pos) {
  if (!h || !d_src_token_pos) return fail(EP_ERR_INVALID_ARG, "NULL argument");
  if (!h->has2d) return fail(EP_ERR_STATE, "no dispatch layout (call ep_dispatch first)");
  *d_src_token_pos = h->w.src_pos;
  return EP_OK;
}

ep_status ep_reset(ep_handle* h, void* stream) {
  (void)stream;
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  h->state = kReady;
  h->has2d = h->hasstd = false;
  return EP_OK;
}

ep_status ep_dispatch_standard_moe(ep_handle* h, const void* x, const float* weights,
                                   const void* scales, const int32_t* indices,
                                   const int32_t* num_tokens, void* stream, ep_std_moe_out* out) {
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  if (!h->g.std_moe) return fail(EP_ERR_INVALID_ARG, "config has standard_moe = 0");
  if (h->state != kReady) return fail(EP_ERR_STATE, "dispatch needs reset() after the previous iteration");
  ep_status s = check_dispatch_inputs(h, x, weights, scales, indices);
  if (s == EP_OK) s = check_tokens(h, num_tokens);
  if (s != EP_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  s = ensure_ready_device(h, st);
  if (s != EP_OK) return s;
  for (int r = 0; r < h->g.R; ++r) h->ntok[r] = num_tokens[r];

  ep::LayoutParams lp;
  fill_layout_common(h, indices, &lp);
  lp.local16 = h->w.local16;
  lp.expert_count = h->w.expert_count;
  lp.expert_offset = h->w.expert_offset;
  lp.rank_rows = h->w.rank_rows;
  lp.rank_base = h->w.rank_base;
  lp.layout_range = h->w.layout_range;
  lp.packed_src_info = h->w.packed_src_info;
  lp.pcap = h->g.pcap;
  lp.chunk_cnt = h->w.chunk_cnt_std;
  lp.chunk_off = h->w.chunk_off_std;
  lp.ticket = h->w.tickets + 1;
  cudaError_t e = ep::launch_layout_std(lp, st);
  if (e != cudaSuccess) return cuda_fail(e, "standard-MoE layout launch");

  ep::DispatchParams dp;
  fill_dispatch_common(h, x, weights, scales, indices, &dp);
  dp.cap = h->g.pcap;
  dp.local16 = h->w.local16;
  dp.chunk_off = h->w.chunk_off_std;
  dp.expert_offset = h->w.expert_offset;
  dp.rank_base = h->w.rank_base;
  dp.src_pos = h->w.packed_src_info;
  dp.row_map = h->w.row_map;
  dp.out_x = h->w.packed_x;
  dp.out_scales = h->w.packed_scales;
  dp.err = h->w.err;
  e = use_bulk_dispatch(h, dp)
          ? ep::launch_dispatch_bulk_copy(dp, true, launch_cfg(h, EP_PHASE_DISPATCH), st)
          : ep::launch_dispatch_std(dp, h->g.quant ? h->cfg.quant_type : 0,
                                    launch_cfg(h, EP_PHASE_DISPATCH), st);
  if (e != cudaSuccess) return cuda_fail(e, "standard-MoE dispatch launch");

  h->state = kDispatched;
  h->has2d = false;
  h->hasstd = true;
  if (out) {
    out->packed_x = h->w.packed_x;
    out->packed_scales = h->g.scale_row_bytes > 0 ? h->w.packed_scales : nullptr;
    out->packed_count = h->w.expert_count;
    out->packed_src_info = h->w.packed_src_info;
    out->packed_layout_range = h->w.layout_range;
    out->expert_offset = h->w.expert_offset;
    out->rank_rows = h->w.rank_rows;
    out->rank_base = h->w.rank_base;
    out->pcap = h->g.pcap;
    out->x_row_bytes = h->g.out_row_bytes;
  }
  return EP_OK;
}

ep_status ep_combine_standard_moe(ep_handle* h, const void* expert_out, const float* weights,
                                  const int32_t* indices, void* out, int32_t call_reset,
                                  void* stream) {
  (void)indices;
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  if (!h->hasstd || h->state == kReady)
    return fail(EP_ERR_STATE, "combine_standard_moe needs a packed layout");
  if (!expert_out || !out) return fail(EP_ERR_INVALID_ARG, "expert_out and out must be non-NULL");
  if (!aligned(expert_out, 16) || !aligned(out, 16))
    return fail(EP_ERR_INVALID_ARG, "expert_out and out must be 16-byte aligned");
  if (h->cfg.weighted_combine && !weights)
    return fail(EP_ERR_INVALID_ARG, "weighted combine needs weights");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ep_status s = ensure_ready_device(h, st);
  if (s != EP_OK) return s;
  const Geometry& g = h->g;
  ep::CombineParams p;
  memset(&p, 0, sizeof(p));
  p.R = g.R; p.Tmax = g.Tmax; p.k = g.k; p.E_r = g.E_r; p.H = g.H;
  for (int r = 0; r < g.R; ++r) p.ntok[r] = h->ntok[r];
  p.cap = g.pcap;
  p.segs_per_token = (g.H + ep::kCombineUnroll * 256 - 1) / (ep::kCombineUnroll * 256);
  p.total_units = (int64_t)g.R * g.Tmax * p.segs_per_token;
  p.weighted = h->cfg.weighted_combine != 0;
  p.y = static_cast<const uint8_t*>(expert_out);
  p.w = weights;
  p.row_map = h->w.row_map;
  p.rank_base = h->w.rank_base;
  p.out = static_cast<uint8_t*>(out);
  p.err = h->w.err;
  cudaError_t e = use_bulk(h, p, true)
                      ? ep::launch_combine_std_bulk(p, h->cfg.combine_dtype,
                                                    h->cfg.combine_out_dtype, launch_cfg(h, EP_PHASE_COMBINE), st)
                      : ep::launch_combine_std(p, h->cfg.combine_dtype, h->cfg.combine_out_dtype,
                                               launch_cfg(h, EP_PHASE_COMBINE), st);
  if (e != cudaSuccess) return cuda_fail(e, "standard-MoE combine launch");
  h->state = kCombined;
  if (call_reset) return ep_reset(h, stream);
  return EP_OK;
}

ep_status ep_convert_dispatch_output(ep_handle* h, const void* dispatch_x,
                                     const int32_t* dispatch_indices, void* stream,
                                     ep_std_moe_out* out) {
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  if (!h->g.std_moe || !h->g.layout2d)
    return fail(EP_ERR_INVALID_ARG, "the conversions need both layouts (standard_moe = 2)");
  if (!h->has2d || h->state != kDispatched)
    return fail(EP_ERR_STATE, "convert_dispatch_output needs a preceding dispatch");
  if (!dispatch_x || !dispatch_indices)
    return fail(EP_ERR_INVALID_ARG, "dispatch_x and dispatch_indices must be non-NULL");
  if (!aligned(dispatch_x, 16)) return fail(EP_ERR_INVALID_ARG, "dispatch_x must be 16-byte aligned");
  if (h->g.scale_row_bytes % 4 != 0)
    return fail(EP_ERR_UNSUPPORTED, "convert needs scale rows that are a multiple of 4 bytes");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ep_status s = ensure_ready_device(h, st);
  if (s != EP_OK) return s;
  const Geometry& g = h->g;
  ep::ConvertParams p;
  memset(&p, 0, sizeof(p));
  p.R = g.R; p.Tmax = g.Tmax; p.k = g.k; p.E_r = g.E_r;
  p.cap = g.cap; p.pcap = g.pcap;
  p.cpr_recv = g.cpr_recv; p.nchunks = g.nchunks_recv;
  p.H = g.H;
  p.row_bytes = g.out_row_bytes;
  p.scale_row_bytes = g.scale_row_bytes;
  p.segs_per_row = (int)((g.out_row_bytes + ep::kCopyUnroll * 512 - 1) / (ep::kCopyUnroll * 512));
  p.total_units = (int64_t)g.R * g.cap * p.segs_per_row;
  p.recv_num_token = h->w.recv_num_token;
  p.recv_idx = dispatch_indices;
  p.src_pos = h->w.src_pos;
  p.recv_x = static_cast<const uint8_t*>(dispatch_x);
  p.recv_scales = h->w.recv_scales;
  p.local16 = h->w.conv_local16;
  p.chunk_cnt = h->w.conv_chunk_cnt;
  p.chunk_off = h->w.conv_chunk_off;
  p.expert_count = h->w.expert_count;
  p.expert_offset = h->w.expert_offset;
  p.rank_rows = h->w.rank_rows;
  p.rank_base = h->w.rank_base;
  p.layout_range = h->w.layout_range;
  p.packed_src_info = h->w.packed_src_info;
  p.row_map = h->w.row_map;
  p.recv_rows = h->w.conv_recv_rows;
  p.packed_x = h->w.packed_x;
  p.packed_scales = h->w.packed_scales;
  p.ticket = h->w.tickets + 2;
  p.err = h->w.err;
  // row_map entries of dropped / foreign slots stay -1
  cudaError_t e = cudaMemsetAsync(h->w.row_map, 0xFF, (size_t)g.R * g.Tmax * g.k * 4, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  e = ep::launch_convert_dispatch(p, g.scale_row_bytes > 0, launch_cfg(h, EP_PHASE_DISPATCH), st);
  if (e != cudaSuccess) return cuda_fail(e, "convert_dispatch_output launch");
  h->hasstd = true;
  if (out) {
    out->packed_x = h->w.packed_x;
    out->packed_scales = g.scale_row_bytes > 0 ? h->w.packed_scales : nullptr;
    out->packed_count = h->w.expert_count;
    out->packed_src_info = h->w.packed_src_info;
    out->packed_layout_range = h->w.layout_range;
    out->expert_offset = h->w.expert_offset;
    out->rank_rows = h->w.rank_rows;
    out->rank_base = h->w.rank_base;
    out->pcap = g.pcap;
    out->x_row_bytes = g.out_row_bytes;
  }
  return EP_OK;
}

ep_status ep_convert_combine_input(ep_handle* h, const void* packed_y, void* combine_in,
                                   void* stream) {
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  if (!h->has2d || !h->hasstd || h->state == kReady)
    return fail(EP_ERR_STATE, "convert_combine_input needs dispatch + convert_dispatch_output");
  if (!packed_y || !combine_in) return fail(EP_ERR_INVALID_ARG, "NULL buffer");
  if (!aligned(packed_y, 16) || !aligned(combine_in, 16))
    return fail(EP_ERR_INVALID_ARG, "buffers must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ep_status s = ensure_ready_device(h, st);
  if (s != EP_OK) return s;
  const Geometry& g = h->g;
  ep::ConvertParams p;
  memset(&p, 0, sizeof(p));
  p.R = g.R; p.Tmax = g.Tmax; p.k = g.k; p.E_r = g.E_r;
  p.cap = g.cap; p.pcap = g.pcap;
  p.H = g.H;
  p.segs_per_row = (g.H + ep::kCombineUnroll * 256 - 1) / (ep::kCombineUnroll * 256);
  p.total_units = (int64_t)g.R * g.cap * p.segs_per_row;
  p.recv_num_token = h->w.recv_num_token;
  p.recv_idx = h->w.recv_idx;
  p.src_pos = h->w.src_pos;
  p.row_map = h->w.row_map;
  p.recv_rows = h->w.conv_recv_rows;
  p.err = h->w.err;
  p.packed_y = static_cast<const uint8_t*>(packed_y);
  p.combine_in = static_cast<uint8_t*>(combine_in);
  // the bulk-copy ring unless the vector kernel is asked for
  const ep::LaunchCfg lc = launch_cfg(h, EP_PHASE_COMBINE);
  cudaError_t e = h->cfg.combine_impl != EP_COMBINE_VECTOR && ep::convert_combine_bulk_supported(p)
                      ? ep::launch_convert_combine_bulk(p, h->cfg.combine_dtype, lc, st)
                      : ep::launch_convert_combine(p, h->cfg.combine_dtype, lc, st);
  if (e != cudaSuccess) return cuda_fail(e, "convert_combine_input launch");
  return EP_OK;
}

ep_status ep_set_launch_config(ep_handle* h, int32_t phase, int32_t impl, int32_t block_num,
                               int32_t warp_num_per_block) {
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  if (phase != EP_PHASE_DISPATCH && phase != EP_PHASE_COMBINE)
    return fail(EP_ERR_INVALID_ARG, "unknown phase %d", phase);
  if (warp_num_per_block > 8) return fail(EP_ERR_INVALID_ARG, "warp_num_per_block must be <= 8");
  if (phase == EP_PHASE_DISPATCH) {
    if (impl < EP_DISPATCH_AUTO || impl > EP_DISPATCH_BULK)
      return fail(EP_ERR_INVALID_ARG, "unknown dispatch_impl %d", impl);
    h->cfg.dispatch_impl = impl;
  } else {
    if (impl < EP_COMBINE_AUTO || impl > EP_COMBINE_BULK)
      return fail(EP_ERR_INVALID_ARG, "unknown combine_impl %d", impl);
    h->cfg.combine_impl = impl;
  }
  h->lc_blocks[phase] = block_num;
  h->lc_warps[phase] = warp_num_per_block;
  return EP_OK;
}

ep_status ep_get_launch_config(const ep_handle* h, int32_t phase, int32_t* impl,
                               int32_t* block_num, int32_t* warp_num_per_block) {
  if (!h || !impl || !block_num || !warp_num_per_block)
    return fail(EP_ERR_INVALID_ARG, "NULL argument");
  if (phase != EP_PHASE_DISPATCH && phase != EP_PHASE_COMBINE)
    return fail(EP_ERR_INVALID_ARG, "unknown phase %d", phase);
  *impl = phase == EP_PHASE_DISPATCH ? h->cfg.dispatch_impl : h->cfg.combine_impl;
  *block_num = h->lc_blocks[phase];
  *warp_num_per_block = h->lc_warps[phase];
  return EP_OK;
}

ep_status ep_selftest_bounded_wait(ep_handle* h, void* stream) {
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ep_status s = ensure_ready_device(h, st);
  if (s != EP_OK) return s;
  cudaError_t e = ep::launch_bounded_wait_selftest(h->w.err, st);
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return EP_OK;
}

ep_status ep_sync(ep_handle* h, void* stream) {
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (h->needs_init) return EP_OK;
  int32_t bits = 0;
  e = cudaMemcpyAsync(&bits, h->w.err, sizeof(bits), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the error flags");
  if (bits == 0) return EP_OK;
  e = cudaMemsetAsync(h->w.err, 0, sizeof(int32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the error flags");
  if (bits & ep::kErrTimeout)
    return fail(EP_ERR_TIMEOUT, "a kernel's bounded wait on a shared-memory barrier gave up");
  if (bits & (ep::kErrIndex | ep::kErrDuplicate))
    return fail(EP_ERR_INVALID_INDEX, "an expert id was outside [-1, %d)%s", h->g.E,
                (bits & ep::kErrDuplicate) ? " or repeated within a token (standard MoE)" : "");
  return fail(EP_ERR_CAPACITY, "packed rows exceed the packed pool of %lld rows",
              (long long)h->g.pcap);
}

}  // extern "C"

// ------------------------------------------------------------------------
// One EP rank per workspace, split send / receive phases (MORI-EP User
// Guide, section 3, "Split dispatch/combine (send + recv)"). The kernels are
// in ep_split.cu; this is the workspace layout, the peer table and the
// per-rank state machine.

namespace {

enum RankState { kRReady = 0, kRSent = 1, kRDispatched = 2, kRCombineSent = 3, kRCombined = 4 };

struct RankCarve {
  int32_t* err;
  unsigned int* tickets;
  uint32_t* mask;            // [Tmax]
  uint8_t* local8;           // [Tmax][R]
  int32_t* chunk_cnt;        // [cpr][R]
  int32_t* chunk_off;        // [cpr][R]
  int32_t* send_cnt;         // [R] own tokens sent to each rank
  int32_t* slot_own;         // [Tmax][R]
  int32_t* send_list;        // [R][Tmax]
  uint8_t* send_x;           // [Tmax][out_row_bytes]
  uint8_t* send_scales;      // [Tmax][scale_row_bytes]
  float* send_w;             // [Tmax][k]
  int32_t* send_idx;         // [Tmax][k]
  int32_t* recv_off;         // [R]
  int32_t* recv_num_token;   // [1]
  int32_t* src_pos;          // [cap]
  uint8_t* recv_x;           // [cap][out_row_bytes]
  uint8_t* recv_scales;      // [cap][scale_row_bytes]
  float* recv_w;             // [cap][k]
  int32_t* recv_idx;         // [cap][k]
  uint8_t* reg_combine_in;   // [cap][H] combine_dtype
  float* comb_w;             // [cap][k] weights given to combine_send
  size_t total;
};

RankCarve carve_rank(const Geometry& g, uint8_t* base) {
  RankCarve c{};
  size_t off = 0;
  const int64_t R = g.R, T = g.Tmax, k = g.k;
  take(base, off, c.err, 4 * sizeof(int32_t));
  take(base, off, c.tickets, 4 * sizeof(unsigned int));
  take(base, off, c.mask, T * 4);
  take(base, off, c.local8, T * R);
  take(base, off, c.chunk_cnt, (size_t)g.cpr * R * 4);
  take(base, off, c.chunk_off, (size_t)g.cpr * R * 4);
  take(base, off, c.send_cnt, R * 4);
  take(base, off, c.slot_own, T * R * 4);
  take(base, off, c.send_list, R * T * 4);
  take(base, off, c.send_x, T * g.out_row_bytes);
  take(base, off, c.send_scales, T * g.scale_row_bytes);
  take(base, off, c.send_w, T * k * 4);
  take(base, off, c.send_idx, T * k * 4);
  take(base, off, c.recv_off, R * 4);
  take(base, off, c.recv_num_token, 4);
  take(base, off, c.src_pos, g.cap * 4);
  take(base, off, c.recv_x, g.cap * g.out_row_bytes);
  take(base, off, c.recv_scales, g.cap * g.scale_row_bytes);
  take(base, off, c.recv_w, g.cap * k * 4);
  take(base, off, c.recv_idx, g.cap * k * 4);
  take(base, off, c.reg_combine_in, g.cap * g.combine_in_row_bytes);
  take(base, off, c.comb_w, g.cap * k * 4);
  c.total = off;
  return c;
}

ep_status make_rank_geometry(const ep_config* cfg, Geometry* g) {
  ep_status s = make_geometry(cfg, g);
  if (s != EP_OK) return s;
  if (g->std_moe)
    return fail(EP_ERR_UNSUPPORTED, "the split send/receive phases use the 2D layout (standard_moe = 0)");
  if (g->scale_row_bytes % 4 != 0)
    return fail(EP_ERR_UNSUPPORTED, "the split phases need scale rows that are a multiple of 4 bytes");
  return EP_OK;
}

}  // namespace

struct ep_rank_handle {
  ep_config cfg;
  Geometry g;
  RankCarve w;
  int rank;
  uint8_t* ws;
  const uint8_t* peers[EP_MAX_WORLD_SIZE];
  bool has_peers;
  int state;
  bool needs_init;
  int ntok;
  int sm_count;
  uint8_t* out;              // combine_send's output buffers, written by combine_recv
  float* out_w;
  bool weighted_w;           // combine_send was given weights
};

namespace {

ep_status rank_ready_device(ep_rank_handle* h, cudaStream_t st) {
  if (h->sm_count == 0) {
    ep_status s = device_sm_count(&h->sm_count);
    if (s != EP_OK) return s;
  }
  if (h->needs_init) {
    cudaError_t e = cudaMemsetAsync(h->w.err, 0, 4 * sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->w.tickets, 0, 4 * sizeof(unsigned int), st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    h->needs_init = false;
  }
  return EP_OK;
}

ep::LaunchCfg rank_launch_cfg(const ep_rank_handle* h) {
  ep::LaunchCfg lc;
  lc.grid_hint = h->cfg.block_num;
  lc.block = (h->cfg.warp_num_per_block > 0 ? h->cfg.warp_num_per_block : 8) * 32;
  lc.sm_count = h->sm_count;
  return lc;
}

ep::SplitPeers rank_peers(const ep_rank_handle* h) {
  ep::SplitPeers pe{};
  for (int r = 0; r < h->g.R; ++r) pe.base[r] = h->peers[r];
  pe.rank = h->rank;
  const uint8_t* b = h->ws;
  auto off = [b](const void* p) { return (int64_t)(static_cast<const uint8_t*>(p) - b); };
  pe.off_send_cnt = off(h->w.send_cnt);
  pe.off_send_list = off(h->w.send_list);
  pe.off_send_x = off(h->w.send_x);
  pe.off_send_scales = off(h->w.send_scales);
  pe.off_send_w = off(h->w.send_w);
  pe.off_send_idx = off(h->w.send_idx);
  pe.off_recv_off = off(h->w.recv_off);
  pe.off_y = off(h->w.reg_combine_in);
  pe.off_w = off(h->w.comb_w);
  return pe;
}

void rank_split_params(const ep_rank_handle* h, ep::SplitParams* p) {
  const Geometry& g = h->g;
  memset(p, 0, sizeof(*p));
  p->R = g.R; p->Tmax = g.Tmax; p->k = g.k; p->E_r = g.E_r; p->E = g.E; p->H = g.H;
  p->ntok = h->ntok;
  p->cap = g.cap;
  p->in_row_bytes = g.in_row_bytes;
  p->out_row_bytes = g.out_row_bytes;
  p->scale_row_bytes = g.scale_row_bytes;
  p->in_scale_row_bytes = g.quant ? 0 : g.in_scale_row_bytes;
  const int64_t step = g.quant ? (int64_t)ep::kQuantUnroll * 512 * 2 : (int64_t)ep::kCopyUnroll * 512;
  p->segs_per_token = (int)((g.in_row_bytes + step - 1) / step);
  p->segs_per_row = (int)((g.out_row_bytes + ep::kCopyUnroll * 512 - 1) / (ep::kCopyUnroll * 512));
  p->total_units = (int64_t)h->ntok * p->segs_per_token;
  p->mask = h->w.mask;
  p->local8 = h->w.local8;
  p->chunk_off = h->w.chunk_off;
  p->slot_own = h->w.slot_own;
  p->send_list = h->w.send_list;
  p->send_x = h->w.send_x;
  p->send_scales = h->w.send_scales;
  p->send_w = h->w.send_w;
  p->send_idx = h->w.send_idx;
  p->recv_x = h->w.recv_x;
  p->recv_scales = h->w.recv_scales;
  p->recv_w = h->w.recv_w;
  p->recv_idx = h->w.recv_idx;
  p->src_pos = h->w.src_pos;
  p->recv_off = h->w.recv_off;
  p->recv_num_token = h->w.recv_num_token;
  p->err = h->w.err;
}

void fill_rank_dispatch_out(const ep_rank_handle* h, ep_dispatch_out* out) {
  if (!out) return;
  out->x = h->w.recv_x;
  out->scales = h->g.scale_row_bytes > 0 ? h->w.recv_scales : nullptr;
  out->weights = h->w.recv_w;
  out->indices = h->w.recv_idx;
  out->recv_num_token = h->w.recv_num_token;
  out->src_token_pos = h->w.src_pos;
  out->cap = h->g.cap;
  out->x_row_bytes = h->g.out_row_bytes;
  out->scale_row_bytes = h->g.scale_row_bytes;
}

}  // namespace

extern "C" {

size_t ep_rank_workspace_size(const ep_config* cfg) {
  Geometry g;
  if (make_rank_geometry(cfg, &g) != EP_OK) return 0;
  return carve_rank(g, nullptr).total;
}

ep_status ep_rank_create(const ep_config* cfg, int32_t rank, void* d_workspace,
                         size_t workspace_bytes, ep_rank_handle** out_handle) {
  if (!out_handle) return fail(EP_ERR_INVALID_ARG, "out_handle is NULL");
  *out_handle = nullptr;
  Geometry g;
  ep_status s = make_rank_geometry(cfg, &g);
  if (s != EP_OK) return s;
  if (rank < 0 || rank >= g.R)
    return fail(EP_ERR_INVALID_ARG, "rank %d outside [0, %d)", rank, g.R);
  const size_t need = carve_rank(g, nullptr).total;
  if (!d_workspace) return fail(EP_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(d_workspace, kAlign)) return fail(EP_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (workspace_bytes < need)
    return fail(EP_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  ep_rank_handle* h = new ep_rank_handle();
  h->cfg = *cfg;
  h->g = g;
  h->rank = rank;
  h->ws = static_cast<uint8_t*>(d_workspace);
  h->w = carve_rank(g, h->ws);
  for (int r = 0; r < EP_MAX_WORLD_SIZE; ++r) h->peers[r] = nullptr;
  h->peers[rank] = h->ws;
  h->has_peers = g.R == 1;
  h->state = kRReady;
  h->needs_init = true;
  h->sm_count = 0;
  *out_handle = h;
  return EP_OK;
}

void ep_rank_destroy(ep_rank_handle* h) { delete h; }

ep_status ep_rank_set_peers(ep_rank_handle* h, void* const* peer_workspaces) {
  if (!h || !peer_workspaces) return fail(EP_ERR_INVALID_ARG, "NULL argument");
  if (h->state != kRReady) return fail(EP_ERR_STATE, "peers can change only between iterations");
  for (int r = 0; r < h->g.R; ++r) {
    if (!peer_workspaces[r]) return fail(EP_ERR_INVALID_ARG, "peer workspace %d is NULL", r);
    if (!aligned(peer_workspaces[r], kAlign))
      return fail(EP_ERR_INVALID_ARG, "peer workspace %d is not 256-byte aligned", r);
  }
  if (peer_workspaces[h->rank] != h->ws)
    return fail(EP_ERR_INVALID_ARG, "entry %d must be this rank's own workspace", h->rank);
  for (int r = 0; r < h->g.R; ++r) h->peers[r] = static_cast<const uint8_t*>(peer_workspaces[r]);
  h->has_peers = true;
  return EP_OK;
}

ep_status ep_dispatch_send(ep_rank_handle* h, const void* x, const float* weights,
                           const void* scales, const int32_t* indices, int32_t num_tokens,
                           void* stream, ep_dispatch_out* out) {
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  if (h->state != kRReady) return fail(EP_ERR_STATE, "dispatch_send needs reset() after the previous iteration");
  const Geometry& g = h->g;
  if (num_tokens < 0 || num_tokens > g.Tmax)
    return fail(EP_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", num_tokens, g.Tmax);
  if (!x || !weights || !indices) return fail(EP_ERR_INVALID_ARG, "x, weights and indices must be non-NULL");
  if (!aligned(x, 16)) return fail(EP_ERR_INVALID_ARG, "x must be 16-byte aligned");
  if (!aligned(weights, 4) || !aligned(indices, 4))
    return fail(EP_ERR_INVALID_ARG, "weights and indices must be 4-byte aligned");
  if (g.quant && scales) return fail(EP_ERR_INVALID_ARG, "scales must be NULL with block quantisation (computed)");
  if (!g.quant && g.in_scale_row_bytes > 0 && !scales) return fail(EP_ERR_INVALID_ARG, "scale_dim > 0 needs a scales array");
  if (scales && !aligned(scales, 4)) return fail(EP_ERR_INVALID_ARG, "scales must be 4-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ep_status s = rank_ready_device(h, st);
  if (s != EP_OK) return s;
  h->ntok = num_tokens;

  // routing layout over this rank's tokens: one source, R destinations
  ep::LayoutParams lp;
  memset(&lp, 0, sizeof(lp));
  lp.R = g.R; lp.Tmax = g.Tmax; lp.k = g.k; lp.E_r = g.E_r; lp.E = g.E;
  lp.cpr = g.cpr; lp.nchunks = g.cpr;
  lp.ntok[0] = num_tokens;
  lp.idx = indices;
  lp.err = h->w.err;
  lp.mask = h->w.mask;
  lp.local8 = h->w.local8;
  lp.recv_num_token = h->w.send_cnt;
  lp.chunk_cnt = h->w.chunk_cnt;
  lp.chunk_off = h->w.chunk_off;
  lp.ticket = h->w.tickets + 0;
  ep::SplitParams sp;
  rank_split_params(h, &sp);
  sp.x = static_cast<const uint8_t*>(x);
  sp.w = weights;
  sp.idx = indices;
  sp.scales_in = static_cast<const uint8_t*>(scales);
  cudaError_t e = ep::launch_layout_2d(lp, st);
  if (e != cudaSuccess) return cuda_fail(e, "routing-layout launch");
  e = ep::launch_split_stage(sp, g.quant ? h->cfg.quant_type : 0, rank_launch_cfg(h), st);
  if (e != cudaSuccess) return cuda_fail(e, "dispatch_send launch");
  h->state = kRSent;
  fill_rank_dispatch_out(h, out);
  return EP_OK;
}

ep_status ep_dispatch_recv(ep_rank_handle* h, void* stream) {
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  if (h->state != kRSent) return fail(EP_ERR_STATE, "dispatch_recv needs a preceding dispatch_send");
  if (!h->has_peers) return fail(EP_ERR_STATE, "peer workspaces are not set (ep_rank_set_peers)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ep_status s = rank_ready_device(h, st);
  if (s != EP_OK) return s;
  ep::SplitParams sp;
  rank_split_params(h, &sp);
  cudaError_t e = ep::launch_split_pull(sp, rank_peers(h), rank_launch_cfg(h), st);
  if (e != cudaSuccess) return cuda_fail(e, "dispatch_recv launch");
  h->state = kRDispatched;
  return EP_OK;
}

ep_status ep_combine_send(ep_rank_handle* h, const void* expert_out, const float* weights,
                          void* out, float* out_weights, void* stream) {
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  if (h->state != kRDispatched) return fail(EP_ERR_STATE, "combine_send needs a completed dispatch (send + recv)");
  if (!out) return fail(EP_ERR_INVALID_ARG, "out must be non-NULL");
  if (!expert_out) expert_out = h->w.reg_combine_in;  // the experts wrote the registered buffer
  if (!aligned(expert_out, 16) || !aligned(out, 16))
    return fail(EP_ERR_INVALID_ARG, "expert_out and out must be 16-byte aligned");
  if ((h->cfg.weighted_combine || out_weights) && !weights)
    return fail(EP_ERR_INVALID_ARG, "weighted combine and out_weights need weights");
  if (weights && !aligned(weights, 4)) return fail(EP_ERR_INVALID_ARG, "weights must be 4-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ep_status s = rank_ready_device(h, st);
  if (s != EP_OK) return s;
  const uint8_t* y = static_cast<const uint8_t*>(expert_out);
  if (y != h->w.reg_combine_in || (weights && weights != h->w.comb_w)) {
    cudaError_t e = ep::launch_split_copy_rows(y, h->w.reg_combine_in, h->g.combine_in_row_bytes,
                                               weights, h->w.comb_w, h->g.k, h->w.recv_num_token,
                                               h->g.cap, rank_launch_cfg(h), st);
    if (e != cudaSuccess) return cuda_fail(e, "combine_send launch");
  }
  h->out = static_cast<uint8_t*>(out);
  h->out_w = out_weights;
  h->weighted_w = weights != nullptr;
  h->state = kRCombineSent;
  return EP_OK;
}

ep_status ep_combine_recv(ep_rank_handle* h, int32_t call_reset, void* stream) {
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  if (h->state != kRCombineSent) return fail(EP_ERR_STATE, "combine_recv needs a preceding combine_send");
  if (!h->has_peers) return fail(EP_ERR_STATE, "peer workspaces are not set (ep_rank_set_peers)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ep_status s = rank_ready_device(h, st);
  if (s != EP_OK) return s;
  const Geometry& g = h->g;
  ep::CombineParams p;
  memset(&p, 0, sizeof(p));
  p.R = g.R; p.Tmax = g.Tmax; p.k = g.k; p.E_r = g.E_r; p.H = g.H;
  p.ntok[0] = h->ntok;
  p.cap = g.cap;
  p.segs_per_token = (g.H + ep::kCombineUnroll * 256 - 1) / (ep::kCombineUnroll * 256);
  p.total_units = (int64_t)h->ntok * p.segs_per_token;
  p.weighted = h->cfg.weighted_combine != 0;
  p.idx = h->w.send_idx;
  p.out = h->out;
  p.out_w = h->out_w;
  p.err = h->w.err;
  cudaError_t e = ep::launch_split_gather(p, rank_peers(h), h->w.slot_own, h->cfg.combine_dtype,
                                          h->cfg.combine_out_dtype, rank_launch_cfg(h), st);
  if (e != cudaSuccess) return cuda_fail(e, "combine_recv launch");
  h->state = kRCombined;
  if (call_reset) h->state = kRReady;
  return EP_OK;
}

ep_status ep_rank_reset(ep_rank_handle* h) {
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  h->state = kRReady;
  return EP_OK;
}

ep_status ep_rank_get_registered_combine_input_buffer(ep_rank_handle* h, void** d_buffer) {
  if (!h || !d_buffer) return fail(EP_ERR_INVALID_ARG, "NULL argument");
  *d_buffer = h->w.reg_combine_in;
  return EP_OK;
}

ep_status ep_rank_get_dispatch_src_token_pos(ep_rank_handle* h, const int32_t** d_src_token_pos) {
  if (!h || !d_src_token_pos) return fail(EP_ERR_INVALID_ARG, "NULL argument");
  if (h->state == kRReady || h->state == kRSent)
    return fail(EP_ERR_STATE, "no received rows yet (dispatch_send, then dispatch_recv)");
  *d_src_token_pos = h->w.src_pos;
  return EP_OK;
}

ep_status ep_rank_sync(ep_rank_handle* h, void* stream) {
  if (!h) return fail(EP_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (h->needs_init) return EP_OK;
  int32_t bits = 0;
  e = cudaMemcpyAsync(&bits, h->w.err, sizeof(bits), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the error flags");
  if (bits == 0) return EP_OK;
  e = cudaMemsetAsync(h->w.err, 0, sizeof(int32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the error flags");
  return fail(EP_ERR_INVALID_INDEX, "an expert id was outside [-1, %d)", h->g.E);
}

}  // extern "C"
