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

// Top-k of one token's logits held 8 per lane (lane l holds experts l + 32 i):
// k rounds of a warp arg-max, larger logit first, lower expert index on ties.
// Two tokens are processed together so that their shuffle chains overlap.
template <int NT>
__device__ __forceinline__ void warp_topk(const float (&v)[NT][8], int npl, int E, int k, int lane,
                                          int (&sel_i)[NT][kMaxTopK], float (&sel_v)[NT][kMaxTopK]) {
  uint32_t taken[NT];
#pragma unroll
  for (int q = 0; q < NT; ++q) taken[q] = 0;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k) {
      float bv[NT];
      int bi[NT];
#pragma unroll
      for (int q = 0; q < NT; ++q) {
        bv[q] = -INFINITY;
        bi[q] = INT_MAX;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int e = lane + 32 * i;
          if (i < npl && e < E && !((taken[q] >> i) & 1u) &&
              (v[q][i] > bv[q] || (v[q][i] == bv[q] && e < bi[q]))) {
            bv[q] = v[q][i];
            bi[q] = e;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int q = 0; q < NT; ++q) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv[q], o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi[q], o);
          if (ov > bv[q] || (ov == bv[q] && oi < bi[q])) {
            bv[q] = ov;
            bi[q] = oi;
          }
        }
      }
#pragma unroll
      for (int q = 0; q < NT; ++q) {
        if ((bi[q] & 31) == lane) taken[q] |= 1u << (bi[q] >> 5);
        sel_i[q][j] = bi[q];
        sel_v[q][j] = bv[q];
      }
    } else {
#pragma unroll
      for (int q = 0; q < NT; ++q) {
        sel_i[q][j] = 0;
        sel_v[q][j] = -INFINITY;
      }
    }
  }
}

__global__ void __launch_bounds__(kRouteThreads) route_topk_kernel(RouteArgs a, int nblk) {
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
  const int npl = (E + 31) >> 5;  // logits per lane (<= 8)
  bool bad = false;

  for (int tl0 = 2 * warp; tl0 < ntok; tl0 += 2 * NW) {
    constexpr int NT = 2;
    float v[NT][8];
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      const int tl = min(tl0 + q, ntok - 1);  // an odd tail repeats the last token
      const float *lt = a.logits + static_cast<size_t>(t0 + tl) * E;
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
        v[q][i] = x;
      }
    }
    int sel_i[NT][kMaxTopK];
    float sel_v[NT][kMaxTopK];
    warp_topk<NT>(v, npl, E, k, lane, sel_i, sel_v);
#pragma unroll
    for (int q = 0; q < NT; ++q) {
      const int tl = tl0 + q;
      if (tl >= ntok) break;
      const size_t sb = static_cast<size_t>(t0 + tl) * k;
      // renormalised weights: exp(l_j - l_max) / sum over the kept set
      const float m = sel_v[q][0];
      float ssum = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (j < k) ssum += expf(sel_v[q][j] - m);
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        if (j < k) {
          if (lane == j) {
            a.topk_idx[sb + j] = sel_i[q][j];
            a.topk_w[sb + j] = expf(sel_v[q][j] - m) / ssum;
            s_pos[tl][sel_i[q][j]] = static_cast<uint8_t>(j);
          }
          if ((sel_i[q][j] >> 5) == lane) word |= 1u << (sel_i[q][j] & 31);
        }
      }
      if (lane < npl) s_mask[tl][lane] = word;
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
