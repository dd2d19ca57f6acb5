// Combine with bulk asynchronous copies (the TMA engine) into a shared-memory
// ring -- same results as combine_2d_kernel / combine_std_kernel, bit for bit.
//
// MORI-EP User Guide, section 3, combine() and section 4,
// combine_standard_moe(); "Choosing an EP API and backend" (EP paths table:
// the combine is a gather, in bf16 or f32). A unit is (source token, 1024-column chunk). A CTA takes
// whole tokens c, c + G, c + 2G, ... (G CTAs), all chunks of each; or, for
// small batches, a contiguous balanced range of units over the present
// tokens (at most one unit more than any other CTA, so a batch of a few
// thousand units has no tail of CTAs with a whole extra token). One
// producer warp per CTA reads the
// token's slot row once (the next token's is prefetched meanwhile), orders
// the token's rows (ascending destination rank; or owner rank then slot for
// the packed layout) and, per chunk, has each lane with a row issue one
// cp.async.bulk of that row chunk into the unit's stage, all completing on
// the stage's mbarrier. Four consumer warps
// wait for the stage, reduce its rows from shared memory in that fixed order
// in f32 (fused multiply-add with the rank's weight when weighted), round
// once and store the output chunk, then release the stage. With four stages
// per CTA the producer runs up to four units ahead, so the latency of one
// unit's slot lookup and row loads overlaps the others' reduction without
// holding any of it in registers. Waits are bounded: on a timeout the kernel
// sets an error bit and returns.
#include "ep_bulk.cuh"
#include "ep_kernels.cuh"

namespace ep {
namespace {

constexpr int kCols = 1024;      // columns of one row chunk (one unit)
constexpr int kStages = 4;       // units in flight per CTA
constexpr int kRows = 8;         // at most 8 rows per unit
constexpr int kConsumers = 4;    // 128 consumer threads x 8 columns = kCols
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int64_t kBalancedMaxUnits = 64;  // units per CTA up to which ranges are balanced

constexpr int esize(int dt) { return dt == EP_DTYPE_BF16 ? 2 : 4; }

struct alignas(16) StageHdr {
  int64_t g;      // source token
  int seg;        // column chunk
  int D;          // rows in the stage; -1 = no token at this position
  int rmin;       // lowest destination rank holding a copy (2D)
  int slmin;      // its receive row
  int pad[2];
  float w[kRows]; // per-row weight (weighted mode)
};

template <int IN>
struct alignas(128) Ring {
  uint8_t data[kStages][kRows][kCols * esize(IN)];
  StageHdr hdr[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
};

template <int OUT>
__device__ __forceinline__ void store8(uint8_t* row, int col, const float f[8]) {
  if (OUT == EP_DTYPE_BF16) {
    st_v4_cs(row + (int64_t)col * 2,
          make_uint4(cvt_bf16x2(f[0], f[1]), cvt_bf16x2(f[2], f[3]), cvt_bf16x2(f[4], f[5]),
                     cvt_bf16x2(f[6], f[7])));
  } else {
    st_v4_cs(row + (int64_t)col * 4, make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                                             __float_as_uint(f[2]), __float_as_uint(f[3])));
    st_v4_cs(row + (int64_t)col * 4 + 16, make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]),
                                                  __float_as_uint(f[6]), __float_as_uint(f[7])));
  }
}

template <int IN>
__device__ __forceinline__ void unpack_smem8(const uint8_t* src, float f[8]) {
  if (IN == EP_DTYPE_BF16) {
    const uint4 v = ld_shared_v4(src);
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
  } else {
    const uint4 a = ld_shared_v4(src), b = ld_shared_v4(src + 16);
    f[0] = __uint_as_float(a.x); f[1] = __uint_as_float(a.y);
    f[2] = __uint_as_float(a.z); f[3] = __uint_as_float(a.w);
    f[4] = __uint_as_float(b.x); f[5] = __uint_as_float(b.y);
    f[6] = __uint_as_float(b.z); f[7] = __uint_as_float(b.w);
  }
}

template <bool STD, int IN, int OUT>
__global__ void __launch_bounds__(kThreads, 3) combine_bulk_kernel(CombineParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Ring<IN>& ring = *reinterpret_cast<Ring<IN>*>(smem_raw);
  constexpr int esz = esize(IN);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ring.full[s], 1);
      mbar_init(&ring.empty[s], kConsumers);
    }
    mbar_init_fence();
  }
  // standard MoE: first pool row of each rank (owner of a pool row = the last
  // rank whose region starts at or before it)
  __shared__ int base[EP_MAX_WORLD_SIZE];
  if (STD && (int)threadIdx.x < p.R) base[threadIdx.x] = __ldg(p.rank_base + threadIdx.x);
  __syncthreads();
  const int segs = p.segs_per_token;
  const int64_t T = p.tok_prefix[p.R];   // present tokens
  // This CTA's units in (token, chunk) order. Balanced: units [u0, u1) over
  // the present tokens. Token-stride: every chunk of tokens c, c + G, ...
  const int64_t U = p.total_units;
  const int64_t u0 = p.balanced ? (int64_t)blockIdx.x * U / gridDim.x : (int64_t)blockIdx.x * segs;
  const int64_t u1 = p.balanced ? (int64_t)(blockIdx.x + 1) * U / gridDim.x : U;
  const int64_t vstep = p.balanced ? 1 : gridDim.x;
  const int64_t nunits =
      p.balanced ? u1 - u0 : (blockIdx.x < T ? (T - blockIdx.x + gridDim.x - 1) / gridDim.x : 0) * segs;
  // global token index of the v-th present token
  auto token_of = [&](int64_t v) -> int64_t {
    int s = 0;
    while (s + 1 < p.R && v >= p.tok_prefix[s + 1]) ++s;
    return (int64_t)s * p.Tmax + (v - p.tok_prefix[s]);
  };

  if (warp == kConsumers) {  // ------------------------------------- producer
    // Slot entry of `lane` for present token v: receive slot on rank `lane`
    // (2D) or packed row of slot `lane` (standard MoE); -1 when absent or
    // past this CTA's units.
    auto mine = [&](int64_t v) { return v < T && v * segs < u1; };
    auto slot_of = [&](int64_t v) -> int {
      if (!mine(v)) return -1;
      const int64_t g = token_of(v);
      if (!STD) return lane < p.R ? __ldg(p.slot_map + g * p.R + lane) : -1;
      return lane < p.k ? __ldg(p.row_map + g * p.k + lane) : -1;
    };
    auto weight_of = [&](int64_t v) -> float {  // standard MoE: router weight of slot `lane`
      if (!STD || !p.weighted || !mine(v) || lane >= p.k) return 0.0f;
      return __ldg(p.w + token_of(v) * p.k + lane);
    };
    int i = 0;
    bool failed = false;
    int64_t v = u0 / segs;
    int sl_next = slot_of(v);
    float w_next = weight_of(v);
    for (; i < nunits && !failed; v += vstep) {
      const int64_t g = token_of(v);
      const int sl = sl_next;
      const float wslot = w_next;
      sl_next = slot_of(v + vstep);   // prefetch the next token's slot row
      w_next = weight_of(v + vstep);
      // rows of this token, their order d and (weighted) their weights
      int d = -1;
      int64_t row = -1;
      float wv = 0.0f;
      const uint32_t m = __ballot_sync(kFull, sl >= 0);
      int rmin = 0, slmin = 0;
      if (!STD) {
        if (sl >= 0) {
          d = __popc(m & lanemask_lt());
          row = (int64_t)lane * p.cap + sl;
          if (p.weighted)
            for (int j = 0; j < p.k; ++j) {
              const int e = __ldg(p.recv_idx + row * p.k + j);
              if (e >= 0 && e / p.E_r == lane) wv = __fadd_rn(wv, __ldg(p.w + row * p.k + j));
            }
        }
        rmin = m ? __ffs(m) - 1 : 0;
        slmin = __shfl_sync(kFull, sl, rmin);
      } else {
        int own = 0;
        while (own + 1 < p.R && sl >= base[own + 1]) ++own;
        const int key = sl >= 0 ? own * 32 + lane : 0x7FFFFFFF;
        int pos = 0;
        for (int q = 0; q < p.k; ++q) pos += __shfl_sync(kFull, key, q) < key;
        if (sl >= 0) {
          d = pos;
          row = sl;
          wv = wslot;
        }
      }
      const int D = __popc(m);
      const int seg0 = (int)(max(u0, v * segs) - v * segs);
      const int seg1 = (int)(min(u1, (v + 1) * segs) - v * segs);
      for (int seg = seg0; seg < seg1; ++seg, ++i) {
        const int st = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        if (i >= kStages && !mbar_wait(&ring.empty[st], ph ^ 1u)) {
          if (lane == 0) atomicOr(p.err, kErrTimeout);
          failed = true;
          break;
        }
        const uint32_t bytes = (uint32_t)(min(kCols, p.H - seg * kCols) * esz);
        StageHdr& h = ring.hdr[st];
        if (lane == 0) {
          h.g = g;
          h.seg = seg;
          h.D = D;
          h.rmin = rmin;
          h.slmin = slmin;
        }
        if (d >= 0) h.w[d] = wv;
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&ring.full[st], (uint32_t)D * bytes);
        __syncwarp();
        if (d >= 0)
          bulk_g2s(ring.data[st][d], p.y + (row * p.H + (int64_t)seg * kCols) * esz, bytes,
                   &ring.full[st]);
      }
    }
    // Do not leave while copies into this CTA's shared memory may be in flight.
    if (lane == 0) {
      for (int j = i - kStages; j < i; ++j) {
        if (j < 0) continue;
        if (!mbar_wait(&ring.full[j % kStages], (uint32_t)(j / kStages) & 1u)) {
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
    const int st = i % kStages;
    const uint32_t ph = (uint32_t)(i / kStages) & 1u;
    if (!mbar_wait(&ring.full[st], ph)) {
      if (lane == 0) atomicOr(p.err, kErrTimeout);
      return;
    }
    const StageHdr& h = ring.hdr[st];
    const int D = h.D, seg = h.seg;
    const int64_t g = h.g;
    const int col = seg * kCols + tid * 8;
    if (col < p.H) {
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
      for (int d = 0; d < kRows; ++d) {
        if (d < D) {
          float f[8];
          unpack_smem8<IN>(ring.data[st][d] + tid * 8 * esz, f);
          const float wd = h.w[d];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            acc[q] = p.weighted ? __fmaf_rn(wd, f[q], acc[q]) : __fadd_rn(acc[q], f[q]);
        }
      }
      store8<OUT>(p.out + g * p.H * esize(OUT), col, acc);
    }
    if (!STD && seg == 0 && p.out_w && warp == 0 && lane < p.k)
      p.out_w[g * p.k + lane] =
          D > 0 ? __ldg(p.w + ((int64_t)h.rmin * p.cap + h.slmin) * p.k + lane) : 0.0f;
    __syncwarp();
    if (lane == 0) mbar_arrive(&ring.empty[st]);
  }
}

template <bool STD>
cudaError_t launch_bulk(const CombineParams& p0, int in_dtype, int out_dtype, const LaunchCfg& lc,
                        cudaStream_t st) {
  CombineParams p = p0;
  p.segs_per_token = (p.H + kCols - 1) / kCols;
  p.tok_prefix[0] = 0;
  for (int s = 0; s < p.R; ++s) p.tok_prefix[s + 1] = p.tok_prefix[s] + p.ntok[s];
  p.total_units = (int64_t)p.tok_prefix[p.R] * p.segs_per_token;
  if (p.total_units == 0) return cudaSuccess;
  const bool ib = in_dtype == EP_DTYPE_BF16, ob = out_dtype == EP_DTYPE_BF16;
  void (*k)(CombineParams) =
      ib ? (ob ? combine_bulk_kernel<STD, EP_DTYPE_BF16, EP_DTYPE_BF16>
               : combine_bulk_kernel<STD, EP_DTYPE_BF16, EP_DTYPE_FP32>)
         : (ob ? combine_bulk_kernel<STD, EP_DTYPE_FP32, EP_DTYPE_BF16>
               : combine_bulk_kernel<STD, EP_DTYPE_FP32, EP_DTYPE_FP32>);
  const size_t smem = ib ? sizeof(Ring<EP_DTYPE_BF16>) : sizeof(Ring<EP_DTYPE_FP32>);
  const int per_sm = ctas_per_sm(k, kThreads, smem);  // also raises the smem limit
  int64_t grid = lc.grid_hint > 0 ? lc.grid_hint : (int64_t)lc.sm_count * per_sm;
  // balanced ranges while a CTA has few units (a token more or less is a
  // large share of its work); whole tokens per CTA otherwise
  p.balanced = p.total_units <= grid * kBalancedMaxUnits;
  if (grid > (p.balanced ? p.total_units : p.tok_prefix[p.R])) grid = p.balanced ? p.total_units : p.tok_prefix[p.R];
  k<<<(unsigned)grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool combine_bulk_supported(const CombineParams& p, bool std_layout) {
  return std_layout ? p.k <= kRows : p.R <= kRows;
}

cudaError_t launch_combine_2d_bulk(const CombineParams& p, int in_dtype, int out_dtype,
                                   const LaunchCfg& lc, cudaStream_t st) {
  return launch_bulk<false>(p, in_dtype, out_dtype, lc, st);
}

cudaError_t launch_combine_std_bulk(const CombineParams& p, int in_dtype, int out_dtype,
                                    const LaunchCfg& lc, cudaStream_t st) {
  return launch_bulk<true>(p, in_dtype, out_dtype, lc, st);
}

}  // namespace ep
