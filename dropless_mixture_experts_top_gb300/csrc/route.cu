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
//   route_topk  : one warp per token.  Top-k by k rounds of warp arg-max
//                 (ties -> lower expert), fp32 renormalised weights, then per
//                 block of 128 tokens an expert histogram and every slot's
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
constexpr int NW = kRouteThreads / 32;

__global__ void __launch_bounds__(kRouteThreads) route_topk_kernel(RouteArgs a, int nblk) {
  __shared__ int32_t s_sel[TB][kMaxTopK];
  __shared__ int32_t s_part[kRouteThreads];
  __shared__ int32_t s_start[kRouteThreads];
  __shared__ int32_t s_cnt[kMaxExperts];
  __shared__ int32_t s_off[kMaxExperts + 1];
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, k = a.k, T = a.T;
  const int t0 = blockIdx.x * TB;
  const int ntok = min(TB, T - t0);
  const int npl = (E + 31) >> 5;  // logits per lane (<= 8)
  bool bad = false;

  for (int tl = warp; tl < ntok; tl += NW) {
    const int t = t0 + tl;
    const float *lt = a.logits + static_cast<size_t>(t) * E;
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      float x = -INFINITY;
      if (i < npl && e < E) {
        x = __ldg(lt + e);
        if (!isfinite(x)) {
          bad = true;
          if (isnan(x)) x = -INFINITY;  // keep the selection well defined
        }
      }
      v[i] = x;
    }
    uint32_t taken = 0;
    int sel_i[kMaxTopK];
    float sel_v[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      sel_i[j] = 0;
      sel_v[j] = -INFINITY;
      if (j < k) {
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int e = lane + 32 * i;
          if (i < npl && e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
            bv = v[i];
            bi = e;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
          }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        sel_i[j] = bi;
        sel_v[j] = bv;
      }
    }
    // renormalised weights: exp(l_j - l_max) / sum over the kept set
    const float m = sel_v[0];
    float ssum = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) ssum += expf(sel_v[j] - m);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k && lane == j) {
        a.topk_idx[static_cast<size_t>(t) * k + j] = sel_i[j];
        a.topk_w[static_cast<size_t>(t) * k + j] = expf(sel_v[j] - m) / ssum;
        s_sel[tl][j] = sel_i[j];
      }
    }
  }
  if (bad) flag_status(a.status, kDevNonfiniteLogit);
  __syncthreads();

  // per-(block, expert) histogram and ranks, in token order
  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    int cnt = 0;
    for (int tl = 0; tl < ntok; ++tl) {
      for (int j = 0; j < k; ++j) {
        if (s_sel[tl][j] == e) {
          a.lrank[static_cast<size_t>(t0 + tl) * k + j] = cnt++;
          break;
        }
      }
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

cudaError_t launch_route_topk(const RouteArgs &a, cudaStream_t s) {
  const int nblk = route_num_blocks(a.T);
  route_topk_kernel<<<nblk, kRouteThreads, 0, s>>>(a, nblk);
  return cudaGetLastError();
}

cudaError_t launch_route_index(const RouteArgs &a, cudaStream_t s) {
  const int n = a.T * a.k;
  route_index_kernel<<<(n + 255) / 256, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
