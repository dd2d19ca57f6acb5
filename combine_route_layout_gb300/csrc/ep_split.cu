// Split dispatch / combine (send + receive phases) for one EP rank per
// workspace, with the other ranks' workspaces reached through device
// pointers (MORI-EP User Guide, section 3, "Split dispatch/combine (send +
// recv)"; section 1, the intra-node kernel type, where ranks exchange tokens
// over peer-to-peer links).
//
// Every rank owns one workspace, carved identically on all ranks, so a
// region of rank s sits at the same offset from s's base pointer. The send
// phases touch only the rank's own memory; the receive phases read the
// peers' memory (pull), so the only ordering the caller provides is that all
// ranks' send phases have completed before any rank's receive phase starts
// (a host barrier after each rank synchronises its stream). No kernel waits
// on another rank.
//
// dispatch_send (rank s): the routing layout over s's own tokens gives each
//   token's destination set, its position in the list of s's tokens sent to
//   each rank r (ascending token order) and the per-destination counts; the
//   stage kernel then writes each token once into s's send buffers (payload
//   or its FP8 / FP4 codes and scales, weights, ids) and the lists of token
//   ids per destination.
// dispatch_recv (rank r): each source's count for r gives the receive
//   offsets (sources ascending, so rows are ordered by (source rank, source
//   token) as in the single-workspace dispatch); the pull kernel copies each
//   receive row from its source's send buffers.
// combine_send (rank r): the expert outputs (and the receive-layout weights)
//   are placed in r's registered buffers, unless the experts wrote them there.
// combine_recv (rank s): for each own token, the rows held by its
//   destination ranks are read from their registered buffers and reduced in
//   ascending rank order, as in the single-workspace combine.
#include "ep_combine_common.cuh"
#include "ep_dispatch_common.cuh"

namespace ep {
namespace {

// ------------------------------------------------------------------ stage
// Unit = (own token, column segment), one warp per unit. Segment payloads go
// to send_x[t]; segment 0 also writes the token's weights, ids, pass-through
// scales, its list position per destination and the destination lists.
template <int QUANT>
__global__ void __launch_bounds__(256, 4) split_stage_kernel(SplitParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  bool waited = false;
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < p.total_units;
       u += nwarps) {
    const int t = (int)(u / p.segs_per_token);
    const int seg = (int)(u - (int64_t)t * p.segs_per_token);
    const uint8_t* src = p.x + (int64_t)t * p.in_row_bytes;
    uint8_t* dst = p.send_x + (int64_t)t * p.out_row_bytes;
    if (QUANT == EP_QUANT_NONE) {
#pragma unroll
      for (int i = 0; i < kCopyUnroll; ++i) {
        const int64_t off = ((int64_t)seg * kCopyUnroll + i) * 512 + lane * 16;
        if (off < p.in_row_bytes) st_v4(dst + off, ld_nc_v4(src + off));
      }
    } else if (QUANT == EP_QUANT_FP4_E2M1_BLOCK32) {
      const int e32 = seg * (kQuantUnroll * 512) + lane * 32;
      if (e32 < p.H) {  // whole 32-element blocks per lane
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = ld_nc_v4(src + (int64_t)e32 * 2 + 16 * i);
        uint4 q;
        float sc;
        quant32_fp4(v, q, sc);
        st_v4(dst + e32 / 2, q);
        reinterpret_cast<float*>(p.send_scales + (int64_t)t * p.scale_row_bytes)[e32 / 32] = sc;
      }
    } else {
      uint4 q[kQuantUnroll];
      float sc[kQuantUnroll];
#pragma unroll
      for (int i = 0; i < kQuantUnroll; ++i) {
        const int e0 = (seg * kQuantUnroll + i) * 512 + lane * 16;
        uint4 a = make_uint4(0, 0, 0, 0), b = a;
        if (e0 < p.H) {
          a = ld_nc_v4(src + (int64_t)e0 * 2);
          b = ld_nc_v4(src + (int64_t)e0 * 2 + 16);
        }
        quant16<true>(a, b, q[i], sc[i]);  // shuffles inside 8-lane groups: all lanes
        if (e0 < p.H) st_v4(dst + e0, q[i]);
      }
      // block scales of the two steps sit in lanes 0, 8, 16, 24
      float* dsc = reinterpret_cast<float*>(p.send_scales + (int64_t)t * p.scale_row_bytes);
#pragma unroll
      for (int i = 0; i < kQuantUnroll; ++i) {
        const int e0 = (seg * kQuantUnroll + i) * 512 + lane * 16;
        if ((lane & 7) == 0 && e0 < p.H) dsc[e0 / 128] = sc[i];
      }
    }
    if (seg != 0) continue;
    // per-token metadata
    if (lane < p.k) {
      p.send_w[(int64_t)t * p.k + lane] = __ldg(p.w + (int64_t)t * p.k + lane);
      p.send_idx[(int64_t)t * p.k + lane] = __ldg(p.idx + (int64_t)t * p.k + lane);
    }
    if (p.in_scale_row_bytes > 0) {
      const uint32_t* s4 = reinterpret_cast<const uint32_t*>(p.scales_in + (int64_t)t * p.in_scale_row_bytes);
      uint32_t* d4 = reinterpret_cast<uint32_t*>(p.send_scales + (int64_t)t * p.scale_row_bytes);
      for (int i = lane; i < p.in_scale_row_bytes / 4; i += 32) d4[i] = __ldg(s4 + i);
    }
    if (!waited) {  // the routing layout is complete and visible past this point
      pdl_wait();
      waited = true;
    }
    const uint32_t m = __ldg(p.mask + t);
    int pos = -1;
    if (lane < p.R && ((m >> lane) & 1u))
      pos = __ldg(p.chunk_off + (int64_t)(t / kChunk) * p.R + lane) +
            __ldg(p.local8 + (int64_t)t * p.R + lane);
    if (lane < p.R) p.slot_own[(int64_t)t * p.R + lane] = pos;
    if (pos >= 0) p.send_list[(int64_t)lane * p.Tmax + pos] = t;
  }
  pdl_wait();  // never finish before the routing layout, even with no work
}

// ------------------------------------------------------------------- pull
// Receive rows of rank `rank`: the count each source s sends here, prefixed
// over s ascending, gives the rows of s; row j = off[s] + i holds token
// send_list_s[rank][i] of s. Unit = (row, 2 KB payload segment), one warp
// per unit; segment 0 also copies the row's scales, weights and ids and
// writes its src_token_pos.
__global__ void __launch_bounds__(256) split_pull_kernel(SplitParams p, SplitPeers pe) {
  __shared__ int cnt[EP_MAX_WORLD_SIZE];
  __shared__ int off[EP_MAX_WORLD_SIZE + 1];
  const int lane = threadIdx.x & 31;
  if ((int)threadIdx.x < p.R)  // every source's count for this rank, loaded in parallel
    cnt[threadIdx.x] =
        __ldcg(reinterpret_cast<const int32_t*>(pe.base[threadIdx.x] + pe.off_send_cnt) + pe.rank);
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int s = 0; s < p.R; ++s) {
      off[s] = acc;
      acc += cnt[s];
    }
    off[p.R] = acc;
  }
  __syncthreads();
  const int total = off[p.R];
  if (blockIdx.x == 0) {
    if ((int)threadIdx.x < p.R) p.recv_off[threadIdx.x] = off[threadIdx.x];
    if (threadIdx.x == 0) p.recv_num_token[0] = total;
  }
  const int segs = p.segs_per_row;
  const int64_t units = (int64_t)total * segs;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < units; u += nwarps) {
    const int j = (int)(u / segs);
    const int seg = (int)(u - (int64_t)j * segs);
    int s = 0;
    while (s + 1 < p.R && j >= off[s + 1]) ++s;
    const uint8_t* peer = pe.base[s];
    const int t = __ldcg(reinterpret_cast<const int32_t*>(peer + pe.off_send_list) +
                         (int64_t)pe.rank * p.Tmax + (j - off[s]));
    const uint8_t* src = peer + pe.off_send_x + (int64_t)t * p.out_row_bytes;
    uint8_t* dst = p.recv_x + (int64_t)j * p.out_row_bytes;
#pragma unroll
    for (int i = 0; i < kCopyUnroll; ++i) {
      const int64_t o = ((int64_t)seg * kCopyUnroll + i) * 512 + lane * 16;
      if (o < p.out_row_bytes) st_v4(dst + o, ld_nc_v4(src + o));
    }
    if (seg != 0) continue;
    if (lane == 0) p.src_pos[j] = s * (p.R * p.Tmax) + t;
    if (lane < p.k) {
      p.recv_w[(int64_t)j * p.k + lane] =
          __ldcg(reinterpret_cast<const float*>(peer + pe.off_send_w) + (int64_t)t * p.k + lane);
      p.recv_idx[(int64_t)j * p.k + lane] =
          __ldcg(reinterpret_cast<const int32_t*>(peer + pe.off_send_idx) + (int64_t)t * p.k + lane);
    }
    if (p.scale_row_bytes > 0) {
      const uint32_t* s4 = reinterpret_cast<const uint32_t*>(peer + pe.off_send_scales +
                                                             (int64_t)t * p.scale_row_bytes);
      uint32_t* d4 = reinterpret_cast<uint32_t*>(p.recv_scales + (int64_t)j * p.scale_row_bytes);
      for (int i = lane; i < p.scale_row_bytes / 4; i += 32) d4[i] = __ldcg(s4 + i);
    }
  }
}

// --------------------------------------------------------- combine_send copy
// Rows [0, recv_num_token) of src (row_bytes each) into dst, and the
// weights rows into dst_w when given; 16 bytes per lane per 512-byte step.
__global__ void __launch_bounds__(256) split_copy_rows_kernel(const uint8_t* src, uint8_t* dst,
                                                             int64_t row_bytes, const float* w,
                                                             float* dst_w, int k,
                                                             const int32_t* count) {
  const int lane = threadIdx.x & 31;
  const int n = __ldcg(count);
  const int segs = (int)((row_bytes + 2047) / 2048);
  const int64_t units = (int64_t)n * segs;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < units; u += nwarps) {
    const int64_t j = u / segs;
    const int seg = (int)(u - j * segs);
    if (src != dst) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t o = ((int64_t)seg * 4 + i) * 512 + lane * 16;
        if (o < row_bytes) st_v4(dst + j * row_bytes + o, ld_nc_v4(src + j * row_bytes + o));
      }
    }
    if (seg == 0 && w && w != dst_w && lane < k) dst_w[j * k + lane] = __ldg(w + j * k + lane);
  }
}

// ------------------------------------------------------------------ gather
// combine_recv of rank pe.rank: unit = (own token, column segment). The
// token's row on destination rank r is r's receive offset for this rank plus
// the token's position in the list sent to r; rows are read from r's
// registered combine input and reduced in ascending r, weighted by the sum
// of the row's weights whose expert r owns (the token's own ids decide
// ownership: they are the ids the row carries).
template <int IN, int OUT, int MAXD>
__global__ void __launch_bounds__(256) split_gather_kernel(CombineParams p, SplitPeers pe,
                                                          const int32_t* slot_own) {
  constexpr int kSlots = MAXD > 0 ? MAXD : EP_MAX_WORLD_SIZE;
  __shared__ int roff[EP_MAX_WORLD_SIZE];
  if ((int)threadIdx.x < p.R)
    roff[threadIdx.x] =
        __ldcg(reinterpret_cast<const int32_t*>(pe.base[threadIdx.x] + pe.off_recv_off) + pe.rank);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t in_row = (int64_t)p.H * dt_size(IN);
  const int64_t out_row = (int64_t)p.H * dt_size(OUT);
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < p.total_units;
       u += nwarps) {
    const int64_t t = u / p.segs_per_token;
    const int seg = (int)(u - t * p.segs_per_token);
    const int sl = lane < p.R ? __ldg(slot_own + t * p.R + lane) : -1;
    const int row = sl >= 0 ? roff[lane] + sl : -1;
    const uint32_t m = __ballot_sync(kFull, sl >= 0);
    const int D = __popc(m);
    const float* wrow = row >= 0 ? reinterpret_cast<const float*>(pe.base[lane] + pe.off_w) +
                                       (int64_t)row * p.k
                                 : nullptr;
    float wr = 0.0f;
    if (p.weighted && row >= 0) {
      for (int j = 0; j < p.k; ++j) {
        const int e = __ldg(p.idx + t * p.k + j);
        if (e >= 0 && e / p.E_r == lane) wr = __fadd_rn(wr, __ldcg(wrow + j));
      }
    }
    if (seg == 0 && p.out_w) {
      const int rmin = m ? __ffs(m) - 1 : 0;
      const float* w0 = reinterpret_cast<const float*>(
          __shfl_sync(kFull, reinterpret_cast<uintptr_t>(wrow), rmin));
      if (lane < p.k) p.out_w[t * p.k + lane] = m ? __ldcg(w0 + lane) : 0.0f;
    }
    const uint8_t* ptr[kSlots];
    float wd[kSlots];
    uint32_t mm = m;
#pragma unroll
    for (int d = 0; d < kSlots; ++d) {
      const int r = mm ? __ffs(mm) - 1 : 0;
      mm &= mm - 1;
      const int rowd = __shfl_sync(kFull, row, r);
      ptr[d] = pe.base[r] + pe.off_y + (int64_t)(rowd < 0 ? 0 : rowd) * in_row;
      wd[d] = __shfl_sync(kFull, wr, r);
    }
    reduce_rows<IN, OUT, MAXD>(p, ptr, wd, D, seg, lane, p.out + t * out_row);
  }
}

}  // namespace

cudaError_t launch_split_stage(const SplitParams& p, int quant, const LaunchCfg& lc,
                               cudaStream_t st) {
  if (p.total_units == 0) {
    // no own tokens: nothing to stage (the layout kernel still ran)
    return cudaSuccess;
  }
  auto k = quant == EP_QUANT_FP8_E4M3_BLOCK128  ? split_stage_kernel<EP_QUANT_FP8_E4M3_BLOCK128>
           : quant == EP_QUANT_FP4_E2M1_BLOCK32 ? split_stage_kernel<EP_QUANT_FP4_E2M1_BLOCK32>
                                                : split_stage_kernel<EP_QUANT_NONE>;
  return launch_pdl(k, auto_grid(k, lc, p.total_units), lc.block, 0, st, p);
}

cudaError_t launch_split_pull(const SplitParams& p, const SplitPeers& pe, const LaunchCfg& lc,
                              cudaStream_t st) {
  // the row count is only known on the device: size the grid for the capacity
  const int64_t units = p.cap * p.segs_per_row;
  const int grid = auto_grid(split_pull_kernel, lc, units);
  split_pull_kernel<<<grid, lc.block, 0, st>>>(p, pe);
  return cudaGetLastError();
}

cudaError_t launch_split_copy_rows(const uint8_t* src, uint8_t* dst, int64_t row_bytes,
                                   const float* w, float* dst_w, int k, const int32_t* count,
                                   int64_t max_rows, const LaunchCfg& lc, cudaStream_t st) {
  const int64_t units = max_rows * ((row_bytes + 2047) / 2048);
  if (units == 0) return cudaSuccess;
  const int grid = auto_grid(split_copy_rows_kernel, lc, units);
  split_copy_rows_kernel<<<grid, lc.block, 0, st>>>(src, dst, row_bytes, w, dst_w, k, count);
  return cudaGetLastError();
}

cudaError_t launch_split_gather(const CombineParams& p, const SplitPeers& pe,
                                const int32_t* slot_own, int in_dtype, int out_dtype,
                                const LaunchCfg& lc, cudaStream_t st) {
  if (p.total_units == 0) return cudaSuccess;
  cudaError_t err = cudaSuccess;
  auto go = [&](auto kernel) {
    kernel<<<auto_grid(kernel, lc, p.total_units), lc.block, 0, st>>>(p, pe, slot_own);
    err = cudaGetLastError();
  };
  const bool ib = in_dtype == EP_DTYPE_BF16, ob = out_dtype == EP_DTYPE_BF16;
  const bool small = p.R <= 8;
  if (ib && ob) small ? go(split_gather_kernel<EP_DTYPE_BF16, EP_DTYPE_BF16, 8>) : go(split_gather_kernel<EP_DTYPE_BF16, EP_DTYPE_BF16, 0>);
  else if (ib) small ? go(split_gather_kernel<EP_DTYPE_BF16, EP_DTYPE_FP32, 8>) : go(split_gather_kernel<EP_DTYPE_BF16, EP_DTYPE_FP32, 0>);
  else if (ob) small ? go(split_gather_kernel<EP_DTYPE_FP32, EP_DTYPE_BF16, 8>) : go(split_gather_kernel<EP_DTYPE_FP32, EP_DTYPE_BF16, 0>);
  else small ? go(split_gather_kernel<EP_DTYPE_FP32, EP_DTYPE_FP32, 8>) : go(split_gather_kernel<EP_DTYPE_FP32, EP_DTYPE_FP32, 0>);
  return err;
}

}  // namespace ep
