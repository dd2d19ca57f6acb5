// Conversions between the 2D receive layout and the standard-MoE packed
// layout (MORI-EP User Guide, section 4: convert_dispatch_output() and
// convert_combine_input()).
//
// convert_dispatch_output: the receive rows of rank r are already in
// (source rank, source token) order, so a row's place inside an expert
// segment is its rank among the rank's receive rows with that expert. A
// layout pass over chunks of 256 receive rows counts rows per local expert
// with per-warp bitmaps, the last CTA scans the chunk counts and lays out the
// 128-row padded segments, a copy pass moves the rows, and a final pass
// derives each (expert, source rank) range by binary search over the sorted
// src_info of the segment. The result equals dispatch_standard_moe().
//
// convert_combine_input: receive row i of rank r becomes the unweighted f32
// sum of the token's packed rows on r (slots ascending), rounded once.
#include <algorithm>

#include "ep_bulk.cuh"
#include "ep_combine_common.cuh"
#include "ep_convert.cuh"
#include "ep_ids.cuh"
#include "ep_kernels.cuh"

namespace ep {
namespace {

constexpr int kWarps = kLayoutThreads / 32;

__device__ bool elect_last(unsigned int* ticket) {
  __shared__ bool last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (last) __threadfence();
  return last;
}

__global__ void __launch_bounds__(kLayoutThreads) conv_layout_kernel(ConvertParams p) {
  extern __shared__ uint32_t dyn[];
  uint32_t* bits = dyn;                                         // [kWarps][E_r]
  uint8_t* pre = reinterpret_cast<uint8_t*>(dyn + kWarps * p.E_r);  // [kWarps][E_r]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x;
  const int r = c / p.cpr_recv;
  const int64_t i = (int64_t)(c % p.cpr_recv) * kChunk + threadIdx.x;
  const bool valid = i < __ldg(p.recv_num_token + r);
  const int64_t row = (int64_t)r * p.cap + i;
  const int E = p.R * p.E_r;

  for (int q = threadIdx.x; q < kWarps * p.E_r; q += blockDim.x) bits[q] = 0u;
  __syncthreads();
  const uint32_t me = 1u << lane;
  int ids[kIdsMax];
  const bool held = valid && load_ids(p.recv_idx + row * p.k, p.k, ids);  // kept for the 2nd pass
  uint32_t counted = 0;  // bit j: slot j holds a row on this rank (written in the 2nd pass)
  if (valid) {
    auto take = [&](int j, int e) {
      if (e < -1 || e >= E) {
        atomicOr(p.err, kErrIndex);
      } else if (e >= 0 && e / p.E_r == r) {
        const uint32_t old = atomicOr(&bits[warp * p.E_r + e % p.E_r], me);
        if (old & me) atomicOr(p.err, kErrDuplicate);
        else counted |= 1u << j;
      }
    };
    if (held) {
#pragma unroll
      for (int j = 0; j < kIdsMax; ++j)
        if (j < p.k) take(j, ids[j]);
    } else {
      for (int j = 0; j < p.k; ++j) take(j, __ldg(p.recv_idx + row * p.k + j));
    }
  }
  __syncthreads();
  for (int el = threadIdx.x; el < p.E_r; el += blockDim.x) {
    int acc = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      pre[w * p.E_r + el] = (uint8_t)acc;
      acc += __popc(bits[w * p.E_r + el]);
    }
    p.chunk_cnt[(int64_t)c * p.E_r + el] = acc;
  }
  __syncthreads();
  if (valid) {
    const uint32_t lt = lanemask_lt();
    auto place = [&](int j, int e) {
      uint16_t v = 0xFFFFu;  // no row on this rank (absent, dropped or repeated id)
      if ((counted >> j) & 1u) {
        const int el = e % p.E_r;
        v = (uint16_t)(pre[warp * p.E_r + el] + __popc(bits[warp * p.E_r + el] & lt));
      }
      p.local16[row * p.k + j] = v;
    };
    if (held) {
#pragma unroll
      for (int j = 0; j < kIdsMax; ++j)
        if (j < p.k) place(j, ids[j]);
    } else {
      for (int j = 0; j < p.k; ++j) place(j, __ldg(p.recv_idx + row * p.k + j));
    }
  }

  if (!elect_last(p.ticket)) return;
  // Last CTA: per (rank, local expert), scan its counts over the rank's
  // receive-row chunks, 16 loads in flight per thread; then the padded
  // segments, each rank's first pool row and the padding rows, with the
  // counts and offsets kept in shared memory (the bitmaps are done).
  int* s_cnt = reinterpret_cast<int*>(dyn);         // [R * E_r]
  int* s_off = s_cnt + p.R * p.E_r;                  // [R * E_r]
  __shared__ int s_base[EP_MAX_WORLD_SIZE];
  __syncthreads();
  for (int q = threadIdx.x; q < p.R * p.E_r; q += blockDim.x) {
    const int rr = q / p.E_r, el = q % p.E_r;
    int run = 0;
    for (int c0 = 0; c0 < p.cpr_recv; c0 += 16) {
      int v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        v[j] = c0 + j < p.cpr_recv
                   ? __ldcg(p.chunk_cnt + (int64_t)(rr * p.cpr_recv + c0 + j) * p.E_r + el)
                   : 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (c0 + j >= p.cpr_recv) break;
        p.chunk_off[(int64_t)(rr * p.cpr_recv + c0 + j) * p.E_r + el] = run;
        run += v[j];
      }
    }
    p.expert_count[q] = run;
    s_cnt[q] = run;
  }
  __syncthreads();
  for (int rr = threadIdx.x; rr < p.R; rr += blockDim.x) {
    int off = 0;
    for (int el = 0; el < p.E_r; ++el) {
      const int q = rr * p.E_r + el;
      p.expert_offset[q] = off;
      s_off[q] = off;
      off += (s_cnt[q] + kPadRows - 1) / kPadRows * kPadRows;
    }
    p.rank_rows[rr] = off;
    s_base[rr] = off;
  }
  __syncthreads();
  // ranks take consecutive regions of the packed pool
  if (threadIdx.x == 0) {
    int64_t base = 0;
    for (int rr = 0; rr < p.R; ++rr) {
      const int rows = s_base[rr];
      s_base[rr] = (int)base;
      p.rank_base[rr] = (int32_t)base;
      base += rows;
    }
    if (base > p.pcap) atomicOr(p.err, kErrCapacity);
  }
  __syncthreads();
  for (int q = warp; q < p.R * p.E_r; q += kWarps) {  // one warp per expert
    const int n = s_cnt[q];
    const int npad = (n + kPadRows - 1) / kPadRows * kPadRows - n;
    const int64_t row0 = (int64_t)s_base[q / p.E_r] + s_off[q] + n;
    for (int j = lane; j < npad; j += 32)
      if (row0 + j < p.pcap) p.packed_src_info[row0 + j] = -1;
  }
  if (threadIdx.x == 0) *p.ticket = 0u;
}

template <bool SCALES>
__global__ void __launch_bounds__(256, 4) conv_copy_kernel(ConvertParams p) {
  const int lane = threadIdx.x & 31;
  const int E = p.R * p.E_r;
  const int64_t stride = (int64_t)p.R * p.Tmax;  // src_token_pos rank stride
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // units run over the present receive rows only: row `row` of the ranks'
  // concatenated rows is row row - pre[r] of rank r
  __shared__ int64_t pre[EP_MAX_WORLD_SIZE + 1];
  if (threadIdx.x == 0) {
    pre[0] = 0;
    for (int r = 0; r < p.R; ++r) {
      const int n = __ldg(p.recv_num_token + r);
      pre[r + 1] = pre[r] + (n < 0 ? 0 : (n > p.cap ? p.cap : n));
    }
  }
  __syncthreads();
  const int64_t units = pre[p.R] * p.segs_per_row;
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < units;
       u += nwarps) {
    const int64_t row = u / p.segs_per_row;
    const int seg = (int)(u - row * p.segs_per_row);
    int r = 0;
    while (r + 1 < p.R && row >= pre[r + 1]) ++r;
    const int64_t i = row - pre[r];
    const int64_t rowg = (int64_t)r * p.cap + i;  // r * cap + i

    const uint8_t* src = p.recv_x + rowg * p.row_bytes;
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int q = 0; q < kCopyUnroll; ++q) {
      const int64_t off = ((int64_t)seg * kCopyUnroll + q) * 512 + lane * 16;
      if (off < p.row_bytes) v[q] = ld_nc_v4(src + off);
    }
    int64_t my_row = -1;
    if (lane < p.k) {
      const int e = __ldg(p.recv_idx + rowg * p.k + lane);
      const int l = __ldg(p.local16 + rowg * p.k + lane);
      if (e >= 0 && e < E && e / p.E_r == r && l != 0xFFFF) {
        const int el = e % p.E_r;
        const int c = r * p.cpr_recv + (int)(i / kChunk);
        const int64_t prow = (int64_t)__ldg(p.rank_base + r) +
                             __ldg(p.expert_offset + r * p.E_r + el) +
                             __ldg(p.chunk_off + (int64_t)c * p.E_r + el) + l;
        if (prow < p.pcap) my_row = prow;
      }
    }
    const uint32_t vm = __ballot_sync(kFull, my_row >= 0);
    if (seg == 0) {
      const int pos = __ldg(p.src_pos + rowg);
      const int64_t g = (pos / stride) * p.Tmax + pos % stride;
      if (my_row >= 0) {
        p.packed_src_info[my_row] = pos;
        p.row_map[g * p.k + lane] = (int32_t)my_row;
      }
      if (lane < p.k) p.recv_rows[rowg * p.k + lane] = (int32_t)my_row;
      if (SCALES) {
        const int nw = p.scale_row_bytes >> 2;
        const uint32_t* ssrc = reinterpret_cast<const uint32_t*>(p.recv_scales + rowg * p.scale_row_bytes);
        for (uint32_t mm = vm; mm; mm &= mm - 1) {
          const int64_t pr = __shfl_sync(kFull, my_row, __ffs(mm) - 1);
          uint32_t* sdst = reinterpret_cast<uint32_t*>(p.packed_scales + pr * p.scale_row_bytes);
          for (int q = lane; q < nw; q += 32) sdst[q] = __ldg(ssrc + q);
        }
      }
    }
    for (uint32_t mm = vm; mm; mm &= mm - 1) {
      const int64_t pr = __shfl_sync(kFull, my_row, __ffs(mm) - 1);
      uint8_t* dst = p.packed_x + pr * p.row_bytes;
#pragma unroll
      for (int q = 0; q < kCopyUnroll; ++q) {
        const int64_t off = ((int64_t)seg * kCopyUnroll + q) * 512 + lane * 16;
        if (off < p.row_bytes) st_v4(dst + off, v[q]);
      }
    }
  }
}

// layout_range[r][el][s] from the sorted src_info of each expert segment:
// thread (r, el, s) finds the first row of source s by binary search; the
// rows of s end where those of s + 1 begin, which the next lane found (a
// shuffle; lane 31 searches for itself), or at the segment's end.
__global__ void conv_range_kernel(ConvertParams p) {
  const int64_t stride = (int64_t)p.R * p.Tmax;
  const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const bool live = q < (int64_t)p.R * p.E_r * p.R;
  int s = 0, n = 0, b = 0;
  const int32_t* seg = nullptr;
  auto lower = [&](int64_t key) {
    int lo = 0, hi = n;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if ((int64_t)seg[mid] < key) lo = mid + 1;
      else hi = mid;
    }
    return lo;
  };
  if (live) {
    s = (int)(q % p.R);
    const int e = (int)(q / p.R);  // r * E_r + el
    seg = p.packed_src_info + (int64_t)p.rank_base[e / p.E_r] + p.expert_offset[e];
    n = p.expert_count[e];
    b = s == 0 ? 0 : lower((int64_t)s * stride);
  }
  const int next_b = __shfl_down_sync(kFull, b, 1);
  if (!live) return;
  const int en = s == p.R - 1 ? n : lane < 31 ? next_b : lower((int64_t)(s + 1) * stride);
  p.layout_range[q] = (int64_t)(((uint64_t)(uint32_t)b << 32) | (uint32_t)(en - b));
}

template <int DT>
__global__ void __launch_bounds__(256) conv_combine_kernel(ConvertParams p) {
  const int lane = threadIdx.x & 31;
  constexpr int esz = DT == EP_DTYPE_BF16 ? 2 : 4;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < p.total_units;
       u += nwarps) {
    const int64_t rowg = u / p.segs_per_row;
    const int seg = (int)(u - rowg * p.segs_per_row);
    const int r = (int)(rowg / p.cap);
    const int64_t i = rowg - (int64_t)r * p.cap;
    if (i >= __ldg(p.recv_num_token + r)) continue;
    // packed rows of this receive row's slots (written by the conversion of
    // the dispatch output): one load, no token lookup in between
    const int prow = lane < p.k ? __ldg(p.recv_rows + rowg * p.k + lane) : -1;
    const uint32_t vm = __ballot_sync(kFull, prow >= 0);
    for (int q = 0; q < kCombineUnroll; ++q) {
      const int e0 = (seg * kCombineUnroll + q) * 256 + lane * 8;
      const bool act = e0 < p.H;  // no early exit: the loop below shuffles
      float acc[8];
#pragma unroll
      for (int z = 0; z < 8; ++z) acc[z] = 0.0f;
      for (uint32_t mm = vm; mm; mm &= mm - 1) {
        const int j = __ffs(mm) - 1;
        const int pr = __shfl_sync(kFull, prow, j);
        if (!act) continue;
        const uint8_t* src = p.packed_y + (int64_t)pr * p.H * esz + (int64_t)e0 * esz;
        float f[8];
        if (DT == EP_DTYPE_BF16) {
          const uint4 v = ld_nc_v4(src);
          f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
          f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
        } else {
          const uint4 a = ld_nc_v4(src), b = ld_nc_v4(src + 16);
          f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y);
          f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
          f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y);
          f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
        }
#pragma unroll
        for (int z = 0; z < 8; ++z) acc[z] = __fadd_rn(acc[z], f[z]);
      }
      if (!act) continue;
      uint8_t* dst = p.combine_in + rowg * p.H * esz + (int64_t)e0 * esz;
      if (DT == EP_DTYPE_BF16) {
        st_v4(dst, make_uint4(cvt_bf16x2(acc[0], acc[1]), cvt_bf16x2(acc[2], acc[3]),
                              cvt_bf16x2(acc[4], acc[5]), cvt_bf16x2(acc[6], acc[7])));
      } else {
        st_v4(dst, make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                              __float_as_uint(acc[2]), __float_as_uint(acc[3])));
        st_v4(dst + 16, make_uint4(__float_as_uint(acc[4]), __float_as_uint(acc[5]),
                                   __float_as_uint(acc[6]), __float_as_uint(acc[7])));
      }
    }
  }
}

// convert_combine_input with bulk asynchronous copies (the TMA engine) into a
// shared-memory ring; the same sums as conv_combine_kernel, bit for bit. A
// unit is (present receive row, 1024-column chunk); CTA b takes present rows
// b, b + G, ... (G CTAs) over all ranks, every chunk of each. One producer
// warp reads a row's packed-row list once (the next row's is fetched
// meanwhile) and, per chunk, has each lane holding a packed row issue one
// cp.async.bulk of that row's chunk into the unit's stage, in slot order;
// four consumer warps sum the stage's rows from shared memory from +0 in
// slot order, round once and store the receive-row chunk. Four stages let
// the producer run up to four units ahead, so row loads are in flight while
// earlier units are summed, without holding them in registers. Waits are
// bounded: on a timeout the kernel sets an error bit and returns.
constexpr int kBCols = 1024;     // columns of one unit
constexpr int kBStages = 4;      // units in flight per CTA
constexpr int kBRows = 8;        // at most 8 packed rows per receive row
constexpr int kBConsumers = 4;   // 128 consumer threads x 8 columns = kBCols
constexpr int kBThreads = (kBConsumers + 1) * 32;

struct alignas(16) ConvStage {
  int64_t rowg;  // receive row r * cap + i
  int seg;       // column chunk
  int D;         // packed rows in the stage
};

template <int DT>
struct alignas(128) ConvRing {
  uint8_t data[kBStages][kBRows][kBCols * dt_size(DT)];
  ConvStage hdr[kBStages];
  uint64_t full[kBStages];
  uint64_t empty[kBStages];
};

template <int DT>
__global__ void __launch_bounds__(kBThreads, 3) conv_combine_bulk_kernel(ConvertParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  ConvRing<DT>& ring = *reinterpret_cast<ConvRing<DT>*>(smem_raw);
  constexpr int esz = dt_size(DT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int64_t pre[EP_MAX_WORLD_SIZE + 1];  // present receive rows before rank r
  if (threadIdx.x == 0) {
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(&ring.full[s], 1);
      mbar_init(&ring.empty[s], kBConsumers);
    }
    mbar_init_fence();
    pre[0] = 0;
    for (int r = 0; r < p.R; ++r) {
      const int n = __ldg(p.recv_num_token + r);
      pre[r + 1] = pre[r] + (n < 0 ? 0 : (n > p.cap ? p.cap : n));
    }
  }
  __syncthreads();
  const int segs = (p.H + kBCols - 1) / kBCols;
  const int64_t rows = pre[p.R];
  const int64_t G = gridDim.x;
  const int64_t nunits = (blockIdx.x < rows ? (rows - blockIdx.x + G - 1) / G : 0) * segs;
  auto rowg_of = [&](int64_t v) -> int64_t {  // v-th present receive row
    int r = 0;
    while (r + 1 < p.R && v >= pre[r + 1]) ++r;
    return (int64_t)r * p.cap + (v - pre[r]);
  };

  if (warp == kBConsumers) {  // ------------------------------------ producer
    auto prow_of = [&](int64_t v) -> int {  // packed row of slot `lane`, -1 if none
      if (v >= rows || lane >= p.k) return -1;
      return __ldg(p.recv_rows + rowg_of(v) * p.k + lane);
    };
    int i = 0;
    bool failed = false;
    int pr_next = prow_of(blockIdx.x);
    for (int64_t v = blockIdx.x; v < rows && !failed; v += G) {
      const int64_t rowg = rowg_of(v);
      const int pr = pr_next;
      pr_next = prow_of(v + G);  // the next row's list is fetched meanwhile
      const uint32_t m = __ballot_sync(kFull, pr >= 0);
      const int d = pr >= 0 ? __popc(m & lanemask_lt()) : -1;  // slot order
      const int D = __popc(m);
      for (int seg = 0; seg < segs; ++seg, ++i) {
        const int st = i % kBStages;
        const uint32_t ph = (uint32_t)(i / kBStages) & 1u;
        if (i >= kBStages && !mbar_wait(&ring.empty[st], ph ^ 1u)) {
          if (lane == 0) atomicOr(p.err, kErrTimeout);
          failed = true;
          break;
        }
        const uint32_t bytes = (uint32_t)(min(kBCols, p.H - seg * kBCols) * esz);
        if (lane == 0) {
          ring.hdr[st].rowg = rowg;
          ring.hdr[st].seg = seg;
          ring.hdr[st].D = D;
          mbar_arrive_expect_tx(&ring.full[st], (uint32_t)D * bytes);
        }
        __syncwarp();
        if (d >= 0)
          bulk_g2s(ring.data[st][d], p.packed_y + ((int64_t)pr * p.H + (int64_t)seg * kBCols) * esz,
                   bytes, &ring.full[st]);
      }
    }
    // Do not leave while copies into this CTA's shared memory may be in flight.
    if (lane == 0) {
      for (int j = i - kBStages; j < i; ++j) {
        if (j < 0) continue;
        if (!mbar_wait(&ring.full[j % kBStages], (uint32_t)(j / kBStages) & 1u)) {
          atomicOr(p.err, kErrTimeout);
          break;
        }
      }
    }
    return;
  }

  // ----------------------------------------------------------------- consumers
  const int tid = threadIdx.x;  // 0 .. 127
  for (int i = 0; i < nunits; ++i) {
    const int st = i % kBStages;
    if (!mbar_wait(&ring.full[st], (uint32_t)(i / kBStages) & 1u)) {
      if (lane == 0) atomicOr(p.err, kErrTimeout);
      return;
    }
    const ConvStage h = ring.hdr[st];
    const int col = h.seg * kBCols + tid * 8;
    if (col < p.H) {
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
      for (int d = 0; d < kBRows; ++d) {
        if (d < h.D) {
          const uint8_t* src = ring.data[st][d] + tid * 8 * esz;
          Raw8<DT> raw;
          raw.a = ld_shared_v4(src);
          if (DT != EP_DTYPE_BF16) raw.b = ld_shared_v4(src + 16);
          float f[8];
          unpack8<DT>(raw, f);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = __fadd_rn(acc[q], f[q]);
        }
      }
      store8<DT>(p.combine_in + h.rowg * p.H * esz, col, acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ring.empty[st]);
  }
}

}  // namespace

bool convert_combine_bulk_supported(const ConvertParams& p) { return p.k <= kBRows; }

cudaError_t launch_convert_combine_bulk(const ConvertParams& p, int dtype, const LaunchCfg& lc,
                                        cudaStream_t st) {
  if (p.total_units == 0) return cudaSuccess;
  const bool bf = dtype == EP_DTYPE_BF16;
  auto k = bf ? conv_combine_bulk_kernel<EP_DTYPE_BF16> : conv_combine_bulk_kernel<EP_DTYPE_FP32>;
  const size_t smem = bf ? sizeof(ConvRing<EP_DTYPE_BF16>) : sizeof(ConvRing<EP_DTYPE_FP32>);
  const int per_sm = ctas_per_sm(k, kBThreads, smem);  // also raises the smem limit
  int64_t grid = lc.grid_hint > 0 ? lc.grid_hint : (int64_t)lc.sm_count * per_sm;
  const int64_t rows = (int64_t)p.R * p.cap;  // upper bound of the present rows
  if (grid > rows) grid = rows;
  k<<<(unsigned)grid, kBThreads, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_convert_dispatch(const ConvertParams& p, bool with_scales,
                                    const LaunchCfg& lc, cudaStream_t st) {
  if (p.nchunks == 0) return cudaSuccess;
  // per-warp bitmaps and prefixes, reused by the last CTA for two int arrays
  // of R * E_r
  const size_t smem = std::max((size_t)kWarps * p.E_r * (sizeof(uint32_t) + 1),
                               (size_t)p.R * p.E_r * 2 * sizeof(int));
  if (smem > 48 * 1024) (void)ctas_per_sm(conv_layout_kernel, kLayoutThreads, smem);
  conv_layout_kernel<<<p.nchunks, kLayoutThreads, smem, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.total_units > 0) {
    auto k = with_scales ? conv_copy_kernel<true> : conv_copy_kernel<false>;
    k<<<auto_grid(k, lc, p.total_units), lc.block, 0, st>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int64_t n = (int64_t)p.R * p.E_r * p.R;
  conv_range_kernel<<<(int)((n + 255) / 256), 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_convert_combine(const ConvertParams& p, int dtype, const LaunchCfg& lc,
                                   cudaStream_t st) {
  if (p.total_units == 0) return cudaSuccess;
  auto k = dtype == EP_DTYPE_BF16 ? conv_combine_kernel<EP_DTYPE_BF16>
                                  : conv_combine_kernel<EP_DTYPE_FP32>;
  k<<<auto_grid(k, lc, p.total_units), lc.block, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace ep
