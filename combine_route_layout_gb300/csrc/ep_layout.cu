// Routing layout (the first half of dispatch).
//
// MORI-EP User Guide, section 3, dispatch(): each token goes to the ranks that
// own its top-k experts (owner = expert / num_experts_per_rank, section 2),
// once per distinct rank (MORI issue 57: a token travels to each owning rank once),
// and dispatch reports recv_num_token. Receive rows are ordered by
// (source rank, source token), which makes every result deterministic.
//
// One CTA handles a chunk of 256 consecutive tokens of one source rank, one
// thread per token. It computes the token's destination set, the chunk's
// per-destination counts (warp ballots) and each token's rank inside the
// chunk, and stores them. The last CTA to finish (elected with one atomic
// ticket after a release fence; no CTA ever waits on another) scans the
// per-chunk counts into per-chunk offsets. The dispatch kernel adds the two.
//
// The standard-MoE variant (User Guide, section 4) counts rows per expert
// instead of per rank (no deduplication), using per-warp expert bitmaps in
// shared memory, and the last CTA also lays out the 128-row padded expert
// segments, the per-source-rank layout ranges and each rank's first row in
// the packed pool the ranks share (the prefix of their padded row counts).
#include "ep_ids.cuh"
#include "ep_kernels.cuh"

namespace ep {
namespace {

constexpr int kWarps = kLayoutThreads / 32;

// Release this CTA's global writes and report whether it finished last.
__device__ bool elect_last_cta(unsigned int* ticket) {
  __shared__ bool last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (last) __threadfence();
  return last;
}

__global__ void __launch_bounds__(kLayoutThreads) layout_2d_kernel(LayoutParams p) {
  pdl_launch_dependents();  // the dispatch kernel may start its independent loads now
  __shared__ int wcnt[kWarps][EP_MAX_WORLD_SIZE];
  __shared__ int wpre[kWarps][EP_MAX_WORLD_SIZE];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x;
  const int s = c / p.cpr;
  const int t = (c % p.cpr) * kChunk + threadIdx.x;
  const bool valid = t < p.ntok[s];
  const int64_t g = (int64_t)s * p.Tmax + t;

  uint32_t m = 0;
  if (valid) {
    const int32_t* row = p.idx + g * p.k;
    auto take = [&](int e) {
      if (e == -1) return;
      if (e < -1 || e >= p.E) {
        atomicOr(p.err, kErrIndex);
        return;
      }
      m |= 1u << (e / p.E_r);
    };
    int ids[kIdsMax];
    if (load_ids(row, p.k, ids)) {
#pragma unroll
      for (int j = 0; j < kIdsMax; ++j)
        if (j < p.k) take(ids[j]);
    } else {
      for (int j = 0; j < p.k; ++j) take(__ldg(row + j));
    }
    p.mask[g] = m;
  }
  for (int r = 0; r < p.R; ++r) {
    const uint32_t b = __ballot_sync(kFull, (m >> r) & 1u);
    if (lane == 0) wcnt[warp][r] = __popc(b);
  }
  __syncthreads();
  if (threadIdx.x < p.R) {
    const int r = threadIdx.x;
    int acc = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      wpre[w][r] = acc;
      acc += wcnt[w][r];
    }
    p.chunk_cnt[(int64_t)c * p.R + r] = acc;
  }
  __syncthreads();
  const uint32_t lt = lanemask_lt();
  for (int r = 0; r < p.R; ++r) {
    const uint32_t b = __ballot_sync(kFull, (m >> r) & 1u);
    if ((m >> r) & 1u) p.local8[g * p.R + r] = (uint8_t)(wpre[warp][r] + __popc(b & lt));
  }

  if (p.no_scan) return;  // small batch: the dispatch kernel sums the chunk counts
  if (!elect_last_cta(p.ticket)) return;
  // Last CTA: one warp per destination rank scans that rank's chunk counts
  // (each lane a contiguous run of chunks), all ranks in parallel.
  const int32_t* __restrict__ cnt = p.chunk_cnt;
  int32_t* __restrict__ off = p.chunk_off;
  const int per = (p.nchunks + 31) / 32;
  for (int r = warp; r < p.R; r += kWarps) {
    const int c0 = min(lane * per, p.nchunks), c1 = min(c0 + per, p.nchunks);
    int sum = 0;
    for (int cc = c0; cc < c1; ++cc) sum += __ldcg(cnt + (int64_t)cc * p.R + r);
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    int ex = incl - sum;
    for (int cc = c0; cc < c1; ++cc) {
      const int v = __ldcg(cnt + (int64_t)cc * p.R + r);
      off[(int64_t)cc * p.R + r] = ex;
      ex += v;
    }
    if (lane == 31) p.recv_num_token[r] = incl;
  }
  if (threadIdx.x == 0) *p.ticket = 0u;
}

__global__ void __launch_bounds__(kLayoutThreads) layout_std_kernel(LayoutParams p) {
  pdl_launch_dependents();
  // bits[w][e]: lanes of warp w whose token selects expert e; pre[w][e]: rows of
  // expert e from warps before w in this chunk.
  extern __shared__ uint32_t dyn[];
  uint32_t* bits = dyn;
  uint8_t* pre = reinterpret_cast<uint8_t*>(dyn + kWarps * p.E);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x;
  const int s = c / p.cpr;
  const int t = (c % p.cpr) * kChunk + threadIdx.x;
  const bool valid = t < p.ntok[s];
  const int64_t g = (int64_t)s * p.Tmax + t;

  for (int i = threadIdx.x; i < kWarps * p.E; i += blockDim.x) bits[i] = 0u;
  __syncthreads();
  const uint32_t me = 1u << lane;
  int ids[kIdsMax];
  const bool held = valid && load_ids(p.idx + g * p.k, p.k, ids);  // ids kept for the 2nd pass
  uint32_t counted = 0;  // bit j: slot j gets a row (its rank is written in the 2nd pass)
  if (valid) {
    const int32_t* row = p.idx + g * p.k;
    auto take = [&](int j, int e) {
      if (e < -1 || e >= p.E) {
        atomicOr(p.err, kErrIndex);
      } else if (e >= 0) {
        const uint32_t old = atomicOr(&bits[warp * p.E + e], me);
        if (old & me) atomicOr(p.err, kErrDuplicate);  // repeated id: later slot dropped
        else counted |= 1u << j;
      }
    };
    if (held) {
#pragma unroll
      for (int j = 0; j < kIdsMax; ++j)
        if (j < p.k) take(j, ids[j]);
    } else {
      for (int j = 0; j < p.k; ++j) take(j, __ldg(row + j));
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    int acc = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      pre[w * p.E + e] = (uint8_t)acc;
      acc += __popc(bits[w * p.E + e]);
    }
    p.chunk_cnt[(int64_t)c * p.E + e] = acc;
  }
  __syncthreads();
  if (valid) {
    const uint32_t lt = lanemask_lt();
    const int32_t* row = p.idx + g * p.k;
    auto place = [&](int j, int e) {
      uint16_t v = 0xFFFFu;  // no row: dropped, invalid or repeated id
      if ((counted >> j) & 1u) v = (uint16_t)(pre[warp * p.E + e] + __popc(bits[warp * p.E + e] & lt));
      p.local16[g * p.k + j] = v;
    };
    if (held) {
#pragma unroll
      for (int j = 0; j < kIdsMax; ++j)
        if (j < p.k) place(j, ids[j]);
    } else {
      for (int j = 0; j < p.k; ++j) place(j, __ldg(row + j));
    }
  }

  if (!elect_last_cta(p.ticket)) return;
  // Last CTA: per expert, scan its counts over the chunks in (source rank,
  // chunk) order, 16 loads in flight per thread; then the padded segment
  // offsets per destination rank, each rank's first pool row, and the
  // padding rows. The counts and offsets stay in shared memory (the expert
  // bitmaps are no longer needed) for the later passes.
  int* s_cnt = reinterpret_cast<int*>(dyn);         // [E]
  int* s_off = s_cnt + p.E;                          // [E]
  __shared__ int s_base[EP_MAX_WORLD_SIZE];
  __syncthreads();                                   // every warp is done with the bitmaps
  const int32_t* __restrict__ cnt = p.chunk_cnt;
  int32_t* __restrict__ coff = p.chunk_off;
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    const int r = e / p.E_r, el = e % p.E_r;
    int run = 0, begin = 0, src = 0, cc = 0;       // chunk c = src * cpr + cc
    for (int c0 = 0; c0 < p.nchunks; c0 += 16) {
      int v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        v[q] = c0 + q < p.nchunks ? __ldcg(cnt + (int64_t)(c0 + q) * p.E + e) : 0;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        if (c0 + q >= p.nchunks) break;
        if (cc == 0) begin = run;
        coff[(int64_t)(c0 + q) * p.E + e] = run;
        run += v[q];
        if (++cc == p.cpr) {  // last chunk of source rank `src`
          p.layout_range[((int64_t)r * p.E_r + el) * p.R + src] =
              (int64_t)(((uint64_t)(uint32_t)begin << 32) | (uint32_t)(run - begin));
          cc = 0;
          ++src;
        }
      }
    }
    p.expert_count[e] = run;
    s_cnt[e] = run;
  }
  __syncthreads();
  for (int r = threadIdx.x; r < p.R; r += blockDim.x) {
    int off = 0;
    for (int el = 0; el < p.E_r; ++el) {
      const int e = r * p.E_r + el;
      p.expert_offset[e] = off;
      s_off[e] = off;
      off += (s_cnt[e] + kPadRows - 1) / kPadRows * kPadRows;
    }
    p.rank_rows[r] = off;
    s_base[r] = off;  // rank r's padded rows; turned into first pool rows below
  }
  __syncthreads();
  // ranks take consecutive regions of the pool shared by all ranks
  if (threadIdx.x == 0) {
    int64_t base = 0;
    for (int r = 0; r < p.R; ++r) {
      const int rows = s_base[r];
      s_base[r] = (int)base;
      p.rank_base[r] = (int32_t)base;
      base += rows;
    }
    if (base > p.pcap) atomicOr(p.err, kErrCapacity);
  }
  __syncthreads();
  // padding rows carry src_info = -1: one warp per expert, a lane per row
  for (int e = warp; e < p.E; e += kWarps) {
    const int n = s_cnt[e];
    const int npad = (n + kPadRows - 1) / kPadRows * kPadRows - n;
    const int64_t row0 = (int64_t)s_base[e / p.E_r] + s_off[e] + n;
    for (int q = lane; q < npad; q += 32)
      if (row0 + q < p.pcap) p.packed_src_info[row0 + q] = -1;
  }
  if (threadIdx.x == 0) *p.ticket = 0u;
}

}  // namespace

cudaError_t launch_layout_2d(const LayoutParams& p, cudaStream_t st) {
  if (p.nchunks == 0) return cudaSuccess;
  layout_2d_kernel<<<p.nchunks, kLayoutThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_layout_std(const LayoutParams& p, cudaStream_t st) {
  if (p.nchunks == 0) return cudaSuccess;
  // per-warp expert bitmaps and prefixes; the last CTA reuses the space for
  // two int arrays of E (8 E bytes <= 40 E bytes)
  const size_t smem = (size_t)kWarps * p.E * (sizeof(uint32_t) + 1);
  if (smem > 48 * 1024) (void)ctas_per_sm(layout_std_kernel, kLayoutThreads, smem);
  layout_std_kernel<<<p.nchunks, kLayoutThreads, smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace ep
