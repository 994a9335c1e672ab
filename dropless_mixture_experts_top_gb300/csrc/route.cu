// route.cu -- router (softmax, top-k, renormalise) and dispatch indices.
//
// Router: a learned router picks the Top-K experts of every token (NVIDIA MoE
// article, intro; the pages do not give its formula -- read as softmax over
// the E logits, keep the k largest, renormalise the kept probabilities).
// Dispatch: tokens are permuted into per-expert groups with data-dependent
// ("ragged") sizes that never leave the device (same article, "Que
// optimizaciones especificas exige el MoE sin descartes": shapes the CPU cannot
// see keep CUDA graphs usable).
//
// Two kernels:
//   route_topk  : the block's 128 tokens' logits staged in shared memory;
//                 four threads per token each keep a sorted top-k list of a
//                 quarter of the experts in registers (branch-free insertion,
//                 ties -> lower expert), merged by two shuffle rounds; fp32
//                 renormalised weights; then per block an expert histogram
//                 and every slot's
//                 rank inside its (block, expert) run.  The last block to
//                 finish (atomic ticket, no spin-wait) scans the histograms:
//                 counts, offsets, and the first row of every (block, expert)
//                 run.  Single pass over the logits.
//   route_index : one thread per slot: row = run base + rank; writes
//                 row_of_slot, slot_of_row and w_row.
// The resulting permutation is expert-major and token-ascending inside an
// expert, so it is unique and reproducible bit for bit.
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int TB = kRouteTokensPerBlock;

constexpr int kQ = kRouteThreads / TB;  // threads per token (4): each scans a quarter of the experts

// (x, xi) ranks before (tv, ti): larger logit first, lower expert index on
// ties; an empty slot (ti == INT_MAX) ranks after everything.
__device__ __forceinline__ bool ranks_before(float x, int xi, float tv, int ti) {
  return x > tv || (x == tv && xi < ti);
}

// Insert (x, xi) into a list sorted by ranks_before, keeping its first KMAX
// entries.  Branch-free: slot j takes slot j-1's entry if x ranks before it,
// else x if x ranks before slot j's entry, else keeps its own.
template <int KMAX>
__device__ __forceinline__ void topk_insert(float (&tv)[KMAX], int (&ti)[KMAX], float x, int xi) {
  bool before[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) before[j] = ranks_before(x, xi, tv[j], ti[j]);
#pragma unroll
  for (int j = KMAX - 1; j > 0; --j) {
    const float v = before[j - 1] ? tv[j - 1] : (before[j] ? x : tv[j]);
    const int ix = before[j - 1] ? ti[j - 1] : (before[j] ? xi : ti[j]);
    tv[j] = v;
    ti[j] = ix;
  }
  if (before[0]) {
    tv[0] = x;
    ti[0] = xi;
  }
}

// The block's logits [ntok, E] (contiguous in memory) into shared memory rows
// of E + 1 floats (the pad keeps the per-token scans free of bank conflicts).
__device__ __forceinline__ void stage_logits(const float *__restrict__ src, int n, int E, float *s_lg) {
  for (int g = 4 * static_cast<int>(threadIdx.x); g < n; g += 4 * kRouteThreads) {
    float v[4];
    if (g + 4 <= n) {
      const float4 q = __ldg(reinterpret_cast<const float4 *>(src + g));
      v[0] = q.x, v[1] = q.y, v[2] = q.z, v[3] = q.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = g + i < n ? __ldg(src + g + i) : 0.f;
    }
    int r = g / E, c = g - r * E;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (g + i < n) s_lg[r * (E + 1) + c] = v[i];
      if (++c == E) {
        c = 0;
        ++r;
      }
    }
  }
}

template <int KMAX>
__global__ void __launch_bounds__(kRouteThreads) route_topk_kernel(RouteArgs a, int nblk) {
  extern __shared__ float s_lg[];                     // [TB][E + 1] this block's logits
  __shared__ uint32_t s_mask[TB][kMaxExperts / 32];  // chosen experts of each token, as bits
  __shared__ uint8_t s_pos[TB][kMaxExperts];         // position j of expert e in the token's list
  __shared__ int32_t s_part[kRouteThreads];
  __shared__ int32_t s_start[kRouteThreads];
  __shared__ int32_t s_cnt[kMaxExperts];
  __shared__ int32_t s_off[kMaxExperts + 1];
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, k = a.k, T = a.T;
  const int t0 = blockIdx.x * TB;
  const int ntok = min(TB, T - t0);
  bool bad = false;

  stage_logits(a.logits + static_cast<size_t>(t0) * E, ntok * E, E, s_lg);
  __syncthreads();

  // Top-k: kQ threads per token (adjacent lanes), each keeps a sorted list of
  // its quarter of the experts, then the lists merge by shuffles.
  {
    const int tl = threadIdx.x / kQ, qq = threadIdx.x % kQ;
    const int per = (E + kQ - 1) / kQ;
    const int e0 = qq * per, e1 = min(E, e0 + per);
    float tv[KMAX];
    int ti[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      tv[j] = -INFINITY;
      ti[j] = INT_MAX;
    }
    if (tl < ntok) {
      const float *row = s_lg + tl * (E + 1);
      for (int e = e0; e < e1; ++e) {
        float x = row[e];
        if (!isfinite(x)) {
          bad = true;
          if (isnan(x)) x = -INFINITY;  // keep the selection well defined
        }
        topk_insert<KMAX>(tv, ti, x, e);
      }
    }
#pragma unroll
    for (int o = 1; o < kQ; o <<= 1) {  // both partners merge the other's list: same result
      float pv[KMAX];
      int pi[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        pv[j] = __shfl_xor_sync(0xffffffffu, tv[j], o);
        pi[j] = __shfl_xor_sync(0xffffffffu, ti[j], o);
      }
#pragma unroll
      for (int j = 0; j < KMAX; ++j) topk_insert<KMAX>(tv, ti, pv[j], pi[j]);
    }
    if (tl < ntok && qq == 0) {
      const size_t sb = static_cast<size_t>(t0 + tl) * k;
      // renormalised weights: exp(l_j - l_max) / sum over the kept set
      const float m = tv[0];
      float ssum = 0.f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k) ssum += expf(tv[j] - m);
      const int npl = (E + 31) >> 5;
      for (int w = 0; w < npl; ++w) s_mask[tl][w] = 0;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k) {
          a.topk_idx[sb + j] = ti[j];
          a.topk_w[sb + j] = expf(tv[j] - m) / ssum;
          s_pos[tl][ti[j]] = static_cast<uint8_t>(j);
          s_mask[tl][ti[j] >> 5] |= 1u << (ti[j] & 31);
        }
      }
    }
  }
  if (bad) flag_status(a.status, kDevNonfiniteLogit);
  __syncthreads();

  // per-(block, expert) histogram and ranks, in token order
  if (threadIdx.x < E) {
    const int e = threadIdx.x, w = e >> 5, b = e & 31;
    int cnt = 0;
#pragma unroll 8
    for (int tl = 0; tl < ntok; ++tl) {
      if ((s_mask[tl][w] >> b) & 1u)
        a.lrank[static_cast<size_t>(t0 + tl) * k + s_pos[tl][e]] = cnt++;
    }
    a.hist[static_cast<size_t>(blockIdx.x) * E + e] = cnt;
  }

  // last block to finish scans all histograms
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.ticket, 1u) == static_cast<unsigned>(nblk - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int P = kRouteThreads / E;  // partial sums per expert (>= 2)
  const int chunk = (nblk + P - 1) / P;
  const int e = threadIdx.x % E, p = threadIdx.x / E;
  const int b0 = p * chunk, b1 = min(nblk, b0 + chunk);
  if (p < P) {
    int s = 0;
#pragma unroll 8
    for (int b = b0; b < b1; ++b) s += __ldcg(a.hist + static_cast<size_t>(b) * E + e);
    s_part[p * E + e] = s;
  }
  __syncthreads();
  if (threadIdx.x < E) {
    int run = 0;
    for (int q = 0; q < P; ++q) {
      s_start[q * E + threadIdx.x] = run;
      run += s_part[q * E + threadIdx.x];
    }
    s_cnt[threadIdx.x] = run;
    a.counts[threadIdx.x] = run;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of counts over experts
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int ee = base + lane;
      const int c = ee < E ? s_cnt[ee] : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (ee < E) s_off[ee] = carry + incl - c;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_off[E] = carry;
  }
  __syncthreads();
  if (threadIdx.x <= E) a.offsets[threadIdx.x] = s_off[threadIdx.x];
  if (p < P) {
    int run = s_off[e] + s_start[p * E + e];
#pragma unroll 8
    for (int b = b0; b < b1; ++b) {
      a.block_base[static_cast<size_t>(b) * E + e] = run;
      run += __ldcg(a.hist + static_cast<size_t>(b) * E + e);
    }
  }
}

__global__ void __launch_bounds__(256) route_index_kernel(RouteArgs a) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  const int nslots = a.T * a.k;
  if (s >= nslots) return;
  const int t = s / a.k;
  const int b = t / TB;
  const int e = a.topk_idx[s];
  const int row = a.block_base[static_cast<size_t>(b) * a.E + e] + a.lrank[s];
  a.row_of_slot[s] = row;
  a.slot_of_row[row] = s;
  a.w_row[row] = a.topk_w[s];
}

}  // namespace

int route_num_blocks(int T) { return (T + TB - 1) / TB; }

template <int KMAX>
cudaError_t launch_topk(const RouteArgs &a, cudaStream_t s) {
  const int nblk = route_num_blocks(a.T);
  const size_t smem = static_cast<size_t>(TB) * (a.E + 1) * sizeof(float);
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {  // room for E = 256
    const cudaError_t e = cudaFuncSetAttribute(route_topk_kernel<KMAX>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               TB * (kMaxExperts + 1) * static_cast<int>(sizeof(float)));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  route_topk_kernel<KMAX><<<nblk, kRouteThreads, smem, s>>>(a, nblk);
  return cudaGetLastError();
}

cudaError_t launch_route_topk(const RouteArgs &a, cudaStream_t s) {
  return a.k <= 8 ? launch_topk<8>(a, s) : launch_topk<kMaxTopK>(a, s);
}

cudaError_t launch_route_index(const RouteArgs &a, cudaStream_t s) {
  const int n = a.T * a.k;
  route_index_kernel<<<(n + 255) / 256, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
