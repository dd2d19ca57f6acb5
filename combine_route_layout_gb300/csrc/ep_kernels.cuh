// Internal declarations shared by the libep translation units: kernel
// parameter blocks, launch helpers and small device primitives written as
// inline PTX for sm_103a.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ep.h"

namespace ep {

constexpr int kChunk = 256;          // source tokens per routing-layout CTA
constexpr int kLayoutThreads = 256;  // one thread per token of the chunk
constexpr int kPadRows = 128;        // standard-MoE segment alignment

// Device error bits, reported by ep_sync.
constexpr int kErrIndex = 1;      // expert id outside [-1, E)
constexpr int kErrDuplicate = 2;  // repeated expert id in one token (standard MoE)
constexpr int kErrCapacity = 4;   // packed rows beyond max_packed_rows_per_rank
constexpr int kErrTimeout = 8;    // a bounded wait on an mbarrier gave up

// ------------------------------------------------------------ parameter blocks

struct LayoutParams {
  int R, Tmax, k, E_r, E;
  int cpr;        // chunks per source rank = ceil(Tmax / kChunk)
  int nchunks;    // R * cpr
  int ntok[EP_MAX_WORLD_SIZE];
  const int32_t* idx;         // [R][Tmax][k]
  // 2D layout
  uint32_t* mask;             // [R*Tmax] destination-rank bitmask
  uint8_t* local8;            // [R*Tmax][R] rank of the token among the chunk's tokens sent to r
  int32_t* recv_num_token;    // [R]
  // standard-MoE layout
  uint16_t* local16;          // [R*Tmax][k] rank among the chunk's rows of that expert; 0xFFFF = none
  int32_t* expert_count;      // [E]
  int32_t* expert_offset;     // [E] segment start within its rank
  int32_t* rank_rows;         // [R] padded rows of each rank
  int32_t* rank_base;         // [R] first pool row of each rank (prefix of rank_rows)
  int64_t* layout_range;      // [R][E_r][R]
  int32_t* packed_src_info;   // [pool rows]
  int64_t pcap;               // rows in the packed pool shared by all ranks
  // shared
  int32_t* chunk_cnt;         // [nchunks][R] (2D) or [nchunks][E] (standard MoE)
  int32_t* chunk_off;         // exclusive prefix over chunks, same shape
  unsigned int* ticket;       // last-CTA election counter (returns to 0)
  int32_t* err;
  int no_scan = 0;            // 2D: leave chunk_off and recv_num_token to the dispatch kernel
};

struct DispatchParams {
  int R, Tmax, k, E_r, E, cpr;
  int ntok[EP_MAX_WORLD_SIZE];
  int64_t cap;                 // receive rows per rank (2D) or packed pool rows (standard MoE)
  int H;
  int64_t in_row_bytes;        // bytes of one source payload row
  int64_t out_row_bytes;       // bytes of one received payload row
  int scale_row_bytes;         // pass-through scale bytes per row (copy mode)
  int segs_per_token;          // work units per token
  int64_t total_units;
  const uint8_t* x;
  const float* w;
  const int32_t* idx;
  const uint8_t* scales_in;
  // layout (from the routing-layout kernel)
  const uint32_t* mask;
  const uint8_t* local8;
  const uint16_t* local16;
  const int32_t* chunk_off;
  const int32_t* expert_offset;
  const int32_t* rank_base;     // standard MoE: first pool row of each rank
  // outputs
  int32_t* slot_map;           // 2D: [R*Tmax][R]
  int32_t* src_pos;            // 2D: [R][cap]; standard MoE: packed_src_info [pool rows]
  int32_t* row_map;            // standard MoE: [R*Tmax][k] global packed row
  uint8_t* out_x;
  uint8_t* out_scales;         // [rows][H/128] f32 (quant) or [rows][scale_row_bytes]
  float* out_w;                // 2D only
  int32_t* out_idx;            // 2D only
  int32_t* err;
  // 2D, small batches (layout run with no_scan): a token's chunk offset is the
  // sum of the earlier chunks' counts, and CTA 0 writes recv_num_token
  const int32_t* chunk_cnt = nullptr;
  int32_t* recv_num_token = nullptr;
};

// Largest chunk count for which the dispatch kernel sums chunk counts itself.
constexpr int kSmallScanChunks = 16;

struct CombineParams {
  int R, Tmax, k, E_r, H;
  int ntok[EP_MAX_WORLD_SIZE];
  int64_t cap;                 // rows per rank of the expert-output buffer
  int segs_per_token;
  int64_t total_units;
  int weighted;
  const uint8_t* y;
  const float* w;              // 2D: receive-layout weights; standard MoE: source weights
  const int32_t* recv_idx;     // 2D: receive-layout expert ids (owner test for weights)
  const int32_t* idx;          // standard MoE: source expert ids
  const int32_t* slot_map;     // 2D
  const int32_t* row_map;      // standard MoE: pool row of each (token, slot)
  const int32_t* rank_base;    // standard MoE: first pool row of each rank
  uint8_t* out;
  float* out_w;
  int32_t* err;
  // bulk kernel: exclusive prefix of ntok (present tokens before rank s), and
  // the work order (1: balanced unit ranges per CTA; 0: whole tokens, strided)
  int tok_prefix[EP_MAX_WORLD_SIZE + 1] = {};
  int balanced = 0;
};

struct ConvertParams {
  int R, Tmax, k, E_r;
  int64_t cap, pcap;           // receive rows per rank; packed pool rows
  int cpr_recv;                // chunks per rank over the receive capacity
  int nchunks;
  int H;
  int64_t row_bytes;
  int scale_row_bytes;
  int segs_per_row;
  int64_t total_units;
  const int32_t* recv_num_token;
  const int32_t* recv_idx;     // [R][cap][k]
  const int32_t* src_pos;      // [R][cap]
  const uint8_t* recv_x;
  const uint8_t* recv_scales;
  uint16_t* local16;           // [R][cap][k]
  int32_t* chunk_cnt;          // [nchunks][E_r]
  int32_t* chunk_off;
  int32_t* expert_count;       // [R][E_r]
  int32_t* expert_offset;
  int32_t* rank_rows;
  int32_t* rank_base;
  int64_t* layout_range;
  int32_t* packed_src_info;
  int32_t* row_map;            // [R*Tmax][k]
  int32_t* recv_rows;          // [R][cap][k] global packed row of each slot of a receive row, -1
  uint8_t* packed_x;
  uint8_t* packed_scales;
  unsigned int* ticket;
  int32_t* err;
  // convert_combine_input
  const uint8_t* packed_y;
  uint8_t* combine_in;
};

// Split send / receive phases, one rank per workspace (ep_split.cu).
struct SplitParams {
  int R, Tmax, k, E_r, E, H;
  int ntok;                    // this rank's tokens
  int64_t cap;                 // receive rows (R * Tmax)
  int64_t in_row_bytes;        // bytes of one source payload row
  int64_t out_row_bytes;       // bytes of one staged / received payload row
  int scale_row_bytes;         // staged / received scale bytes per row (0 = none)
  int in_scale_row_bytes;      // pass-through input scale bytes per row
  int segs_per_token;          // stage units per token
  int segs_per_row;            // pull units per receive row (2 KB each)
  int64_t total_units;         // stage units
  // send side (this rank's own memory)
  const uint8_t* x;
  const float* w;
  const int32_t* idx;
  const uint8_t* scales_in;
  const uint32_t* mask;        // [Tmax] destination ranks of each own token
  const uint8_t* local8;       // [Tmax][R]
  const int32_t* chunk_off;    // [cpr][R]
  int32_t* slot_own;           // [Tmax][R] position in the list sent to r, or -1
  int32_t* send_list;          // [R][Tmax] own token ids sent to r, ascending
  uint8_t* send_x;             // [Tmax][out_row_bytes]
  uint8_t* send_scales;        // [Tmax][scale_row_bytes]
  float* send_w;               // [Tmax][k]
  int32_t* send_idx;           // [Tmax][k]
  // receive side
  uint8_t* recv_x;             // [cap][out_row_bytes]
  uint8_t* recv_scales;
  float* recv_w;
  int32_t* recv_idx;
  int32_t* src_pos;            // [cap]
  int32_t* recv_off;           // [R] first receive row of each source
  int32_t* recv_num_token;     // [1]
  int32_t* err;
};

// Every rank's workspace base and the byte offsets of the regions peers read
// (identical on all ranks: same config, same carve).
struct SplitPeers {
  const uint8_t* base[EP_MAX_WORLD_SIZE];
  int rank;
  int64_t off_send_cnt, off_send_list, off_send_x, off_send_scales, off_send_w, off_send_idx;
  int64_t off_recv_off;        // receive offsets per source
  int64_t off_y;               // registered combine input
  int64_t off_w;               // combine weights in receive layout
};

// ------------------------------------------------------------------ launchers
// Each returns the cudaError_t of its launch.

struct LaunchCfg {
  int grid_hint;  // CTAs requested by the caller; <= 0: one full wave
  int block;      // threads per CTA (multiple of 32, <= 256)
  int sm_count;
};

// Resident CTAs per SM for (kernel, block, dynamic smem) on the current
// device; raises the kernel's dynamic shared-memory limit first when smem
// exceeds the default. Cached after the first query, so a launch costs no
// occupancy calculation.
int ctas_per_sm(const void* kernel, int block, size_t smem);

template <typename Kernel>
inline int ctas_per_sm(Kernel kernel, int block, size_t smem = 0) {
  return ctas_per_sm(reinterpret_cast<const void*>(kernel), block, smem);
}

// CTAs for a grid-stride kernel over `units` warp-sized work units: the
// caller's request, else as many CTAs as fit on the GPU at once, never more
// than the units need.
template <typename Kernel>
inline int auto_grid(Kernel kernel, const LaunchCfg& lc, int64_t units, size_t smem = 0) {
  const int64_t warps = lc.block / 32;
  const int64_t need = (units + warps - 1) / warps;
  int64_t grid = lc.grid_hint;
  if (grid <= 0) grid = (int64_t)lc.sm_count * ctas_per_sm(kernel, lc.block, smem);
  if (grid > need) grid = need;
  return grid < 1 ? 1 : (int)grid;
}

cudaError_t launch_layout_2d(const LayoutParams& p, cudaStream_t st);
cudaError_t launch_layout_std(const LayoutParams& p, cudaStream_t st);
// quant: 0 = copy, EP_QUANT_FP8_E4M3_BLOCK128 or EP_QUANT_FP4_E2M1_BLOCK32.
cudaError_t launch_dispatch_2d(const DispatchParams& p, int quant, const LaunchCfg& lc,
                               cudaStream_t st);
cudaError_t launch_dispatch_std(const DispatchParams& p, int quant, const LaunchCfg& lc,
                                cudaStream_t st);
cudaError_t launch_combine_2d(const CombineParams& p, int in_dtype, int out_dtype,
                              const LaunchCfg& lc, cudaStream_t st);
cudaError_t launch_combine_std(const CombineParams& p, int in_dtype, int out_dtype,
                               const LaunchCfg& lc, cudaStream_t st);
// Bulk-copy (TMA engine) combine; same results as the vector kernels. Needs
// at most 8 rows per token (world_size <= 8, or top-k <= 8 for the packed layout).
bool combine_bulk_supported(const CombineParams& p, bool std_layout);
cudaError_t launch_combine_2d_bulk(const CombineParams& p, int in_dtype, int out_dtype,
                                   const LaunchCfg& lc, cudaStream_t st);
cudaError_t launch_combine_std_bulk(const CombineParams& p, int in_dtype, int out_dtype,
                                    const LaunchCfg& lc, cudaStream_t st);
// One kernel whose bounded mbarrier wait times out (about 1 s) and sets
// kErrTimeout in *err.
cudaError_t launch_bounded_wait_selftest(int32_t* err, cudaStream_t st);

// Copy-mode dispatch with bulk copies (TMA); same results as the vector
// kernel. Needs source rows of at most 48 KB.
bool dispatch_bulk_supported(const DispatchParams& p);
cudaError_t launch_dispatch_bulk_copy(const DispatchParams& p, bool std_layout,
                                      const LaunchCfg& lc, cudaStream_t st);
cudaError_t launch_convert_dispatch(const ConvertParams& p, bool with_scales,
                                    const LaunchCfg& lc, cudaStream_t st);
cudaError_t launch_convert_combine(const ConvertParams& p, int dtype, const LaunchCfg& lc,
                                   cudaStream_t st);

// Split phases (ep_split.cu). quant as for launch_dispatch_2d.
cudaError_t launch_split_stage(const SplitParams& p, int quant, const LaunchCfg& lc,
                               cudaStream_t st);
cudaError_t launch_split_pull(const SplitParams& p, const SplitPeers& pe, const LaunchCfg& lc,
                              cudaStream_t st);
// Rows [0, *count) of src into dst (skipped when src == dst) and, when w is
// given and differs from dst_w, their k weights into dst_w.
cudaError_t launch_split_copy_rows(const uint8_t* src, uint8_t* dst, int64_t row_bytes,
                                   const float* w, float* dst_w, int k, const int32_t* count,
                                   int64_t max_rows, const LaunchCfg& lc, cudaStream_t st);
cudaError_t launch_split_gather(const CombineParams& p, const SplitPeers& pe,
                                const int32_t* slot_own, int in_dtype, int out_dtype,
                                const LaunchCfg& lc, cudaStream_t st);

// Record `msg` as the calling thread's ep_last_error() text; returns `st`.
ep_status record_error(ep_status st, const char* msg);

// Work-unit geometry used by the launchers and the host library alike.
constexpr int kCopyUnroll = 4;       // 16-byte vectors per lane per copy unit
constexpr int kQuantUnroll = 2;      // 512-element steps per quantisation unit
#ifndef EP_COMBINE_UNROLL
#define EP_COMBINE_UNROLL 2
#endif
constexpr int kCombineUnroll = EP_COMBINE_UNROLL;  // 256-element steps per combine unit

// Launch `kernel` with programmatic stream serialization, so it may begin
// while the previous kernel in the stream is still running (it waits with
// griddepcontrol.wait before reading that kernel's outputs).
template <typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Args...), int grid, int block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace ep

// ---------------------------------------------------------------- device PTX
#ifdef __CUDACC__
namespace ep {

constexpr unsigned kFull = 0xFFFFFFFFu;  // every lane of a warp

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Streaming store (evict-first): for outputs this kernel will not read again.
__device__ __forceinline__ void st_v4_cs(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Two f32 -> two OCP E4M3 codes, round to nearest even, saturating to +-448.
// Returns lo in bits 0..7 and hi in bits 8..15.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight f32 -> eight OCP E2M1 codes, round to nearest even, saturating to
// +-6; byte k holds elements 2k (low nibble) and 2k+1 (high nibble).
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float f[8]) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(r)
      : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7]));
  return r;
}

// Two f32 -> two bf16 (round to nearest even); lo in bits 0..15.
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Programmatic dependent launch: let the next kernel in the stream start
// (it must call pdl_wait before touching this kernel's outputs) ...
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// ... and, in that next kernel, wait until the previous grid has finished and
// its writes are visible. A no-op when the kernel was launched without PDL.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace ep
#endif
