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
//   route_topk  : the block's 128 tokens' logits staged in shared memory (all
//                 of a thread's loads issued before the first store);
//                 four threads per token each take every fourth expert, sort
//                 them KMAX at a time with a bitonic network and keep the best
//                 KMAX (bitonic top-k merge); the four lists merge by two
//                 shuffle rounds.  Ties -> lower expert.  fp32 renormalised
//                 weights.  Every token's chosen experts set one bit in a
//                 per-expert bitmask over the block's tokens, so a slot's rank
//                 inside its (block, expert) run, in token order, is a
//                 popcount and the block's expert histogram a sum of them.
//                 Single pass over the logits.
//   route_index : one block per route block: every block sums the histogram
//                 columns (below its own row, and in total), scans the totals
//                 over experts (counts, offsets; block 0 writes them), and
//                 writes its slots' rows: row = offsets[e] + the rows of
//                 expert e in earlier blocks + rank; row_of_slot, slot_of_row,
//                 w_row.  The kernel boundary is the only grid-wide wait.
// The resulting permutation is expert-major and token-ascending inside an
// expert, so it is unique and reproducible bit for bit.
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int TB = kRouteTokensPerBlock;

constexpr int kQ = kRouteThreads / TB;      // threads per token (4): each takes every kQ-th expert
constexpr int kTokPerWarp = 32 / kQ;        // tokens of one warp (8); a token's threads are kTokPerWarp lanes apart
constexpr int kMaskWords = TB / 32;         // words of a per-expert token bitmask
constexpr int kLoadBatch = 8;               // float4 loads a thread has in flight while staging
constexpr int kHistLoads = 32;              // histogram loads a route_index thread has in flight

// (x, xi) ranks before (y, yi): larger logit first, lower expert index on
// ties; an empty slot (index INT_MAX, value -inf) ranks after everything.
__device__ __forceinline__ bool ranks_before(float x, int xi, float y, int yi) {
  return x > y || (x == y && xi < yi);
}

// Order the pair so that slot a ranks before slot b.
__device__ __forceinline__ void order_pair(float &av, int &ai, float &bv, int &bi) {
  const bool sw = ranks_before(bv, bi, av, ai);
  const float tv = sw ? bv : av;
  const int ti = sw ? bi : ai;
  bv = sw ? av : bv;
  bi = sw ? ai : bi;
  av = tv;
  ai = ti;
}

// Bitonic sorting network over N (a power of two) entries: afterwards entry 0
// ranks first.  Blocks of `size` entries alternate direction until the last
// stage, where every pair orders first-before-second.
template <int N>
__device__ __forceinline__ void bitonic_sort(float (&v)[N], int (&ix)[N]) {
#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int st = size >> 1; st > 0; st >>= 1) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
        if ((i & st) == 0) {
          if ((i & size) == 0)
            order_pair(v[i], ix[i], v[i + st], ix[i + st]);
          else
            order_pair(v[i + st], ix[i + st], v[i], ix[i]);
        }
      }
    }
  }
}

// a <- the best N of a and b, sorted; both sorted on entry.  Entry i of a
// against entry N-1-i of b keeps the better one: the result holds the N best
// of both and is bitonic, and a cascade of half-cleaners sorts it.
template <int N>
__device__ __forceinline__ void merge_best(float (&av)[N], int (&ai)[N], const float (&bv)[N],
                                           const int (&bi)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const bool tb = ranks_before(bv[N - 1 - i], bi[N - 1 - i], av[i], ai[i]);
    av[i] = tb ? bv[N - 1 - i] : av[i];
    ai[i] = tb ? bi[N - 1 - i] : ai[i];
  }
#pragma unroll
  for (int st = N >> 1; st > 0; st >>= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if ((i & st) == 0) order_pair(av[i], ai[i], av[i + st], ai[i + st]);
  }
}

// The block's logits [n / E, E] (contiguous in memory, 16-byte aligned: the
// block's first token is a multiple of 128) into shared memory rows of S
// floats.  Each thread issues kLoadBatch 16-byte loads before its first
// store, so the block waits for one round trip to memory, not one per load.
// A NaN is staged as -inf (the selection stays well defined); returns whether
// this thread saw a non-finite logit.
__device__ __forceinline__ float nan_to_ninf(float x, bool &bad) {
  bad |= !isfinite(x);
  return x != x ? -INFINITY : x;
}

__device__ __forceinline__ bool stage_logits(const float *__restrict__ src, int n, int E, int S,
                                             float *s_lg) {
  bool bad = false;
  for (int base = 0; base < n; base += 4 * kRouteThreads * kLoadBatch) {
    float4 q[kLoadBatch];
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      const int g = base + 4 * (static_cast<int>(threadIdx.x) + u * kRouteThreads);
      if (g + 4 <= n) {
        q[u] = __ldg(reinterpret_cast<const float4 *>(src + g));
      } else {
        q[u].x = g < n ? __ldg(src + g) : 0.f;
        q[u].y = g + 1 < n ? __ldg(src + g + 1) : 0.f;
        q[u].z = g + 2 < n ? __ldg(src + g + 2) : 0.f;
        q[u].w = g + 3 < n ? __ldg(src + g + 3) : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      q[u].x = nan_to_ninf(q[u].x, bad);
      q[u].y = nan_to_ninf(q[u].y, bad);
      q[u].z = nan_to_ninf(q[u].z, bad);
      q[u].w = nan_to_ninf(q[u].w, bad);
    }
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      const int g = base + 4 * (static_cast<int>(threadIdx.x) + u * kRouteThreads);
      if (g >= n) break;
      int r = g / E, c = g - r * E;
      if ((E & 3) == 0) {  // the four stay in one row; rows start 16-byte aligned
        *reinterpret_cast<float4 *>(s_lg + r * S + c) = q[u];
      } else {
        const float v[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (g + i < n) s_lg[r * S + c] = v[i];
          if (++c == E) {
            c = 0;
            ++r;
          }
        }
      }
    }
  }
  return bad;
}

// Shared-memory row stride of the staged logits: E + 4 floats keeps rows
// 16-byte aligned and puts the 8 tokens x 4 quarters of a warp's reads
// (token tl, expert q + 4m) on distinct banks when E is a multiple of 32.
__host__ __device__ constexpr int logit_stride(int E) { return E + 4; }

template <int KMAX>
__global__ void __launch_bounds__(kRouteThreads) route_topk_kernel(RouteArgs a) {
  extern __shared__ __align__(16) float s_lg[];           // [TB][E + 4] this block's logits
  __shared__ uint32_t s_emask[kMaxExperts][kMaskWords];  // tokens of this block that chose expert e
  __shared__ uint8_t s_slot_e[TB * kMaxTopK];            // expert of each of the block's slots

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, k = a.k, T = a.T;
  const int S = logit_stride(E);
  const int t0 = blockIdx.x * TB;
  const int ntok = min(TB, T - t0);

  for (int i = threadIdx.x; i < E * kMaskWords; i += kRouteThreads) (&s_emask[0][0])[i] = 0u;
  const bool bad = stage_logits(a.logits + static_cast<size_t>(t0) * E, ntok * E, E, S, s_lg);
  __syncthreads();

  // Top-k of token tl by its kQ threads (lanes kTokPerWarp apart): quarter qq
  // takes experts qq, qq + kQ, qq + 2kQ, ...
  {
    const int tl = warp * kTokPerWarp + lane % kTokPerWarp, qq = lane / kTokPerWarp;
    const int nm = tl < ntok ? (E - qq + kQ - 1) / kQ : 0;  // this quarter's experts
    const float *row = s_lg + tl * S;
    float tv[KMAX];
    int ti[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      tv[j] = -INFINITY;
      ti[j] = INT_MAX;
    }
    for (int m0 = 0; m0 < nm; m0 += KMAX) {
      float cv[KMAX];
      int ci[KMAX];
#pragma unroll
      for (int u = 0; u < KMAX; ++u) {
        const int m = m0 + u, e = qq + kQ * m;
        cv[u] = m < nm ? row[e] : -INFINITY;
        ci[u] = m < nm ? e : INT_MAX;
      }
      bitonic_sort<KMAX>(cv, ci);
      if (m0 == 0) {  // the first chunk is the running list
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          tv[j] = cv[j];
          ti[j] = ci[j];
        }
      } else {
        merge_best<KMAX>(tv, ti, cv, ci);
      }
    }
#pragma unroll
    for (int o = kTokPerWarp; o < 32; o <<= 1) {  // both partners merge the same two lists
      float pv[KMAX];
      int pi[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        pv[j] = __shfl_xor_sync(0xffffffffu, tv[j], o);
        pi[j] = __shfl_xor_sync(0xffffffffu, ti[j], o);
      }
      merge_best<KMAX>(tv, ti, pv, pi);
    }
    if (tl < ntok) {
      const size_t sb = static_cast<size_t>(t0 + tl) * k;
      // renormalised weights: exp(l_j - l_max) / sum over the kept set
      const float m = tv[0];
      float ssum = 0.f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k) ssum += expf(tv[j] - m);
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k && j % kQ == qq) {  // the token's kQ threads share its k slots
          a.topk_idx[sb + j] = ti[j];
          a.topk_w[sb + j] = expf(tv[j] - m) / ssum;
          s_slot_e[tl * k + j] = static_cast<uint8_t>(ti[j]);
          atomicOr(&s_emask[ti[j]][tl >> 5], 1u << (tl & 31));
        }
      }
    }
  }
  if (bad) flag_status(a.status, kDevNonfiniteLogit);
  __syncthreads();

  // rank of every slot inside its (block, expert) run: the run's tokens before it
  for (int sl = threadIdx.x; sl < ntok * k; sl += kRouteThreads) {
    const int tl = sl / k;
    const uint32_t *mk = s_emask[s_slot_e[sl]];
    int r = __popc(mk[tl >> 5] & ((1u << (tl & 31)) - 1u));
    for (int w = 0; w < (tl >> 5); ++w) r += __popc(mk[w]);
    a.lrank[static_cast<size_t>(t0) * k + sl] = r;
  }
  if (threadIdx.x < E) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < kMaskWords; ++w) c += __popc(s_emask[threadIdx.x][w]);
    a.hist[static_cast<size_t>(blockIdx.x) * E + threadIdx.x] = c;
  }
}

__global__ void __launch_bounds__(kRouteThreads) route_index_kernel(RouteArgs a, int nblk) {
  __shared__ int32_t s_below[kRouteThreads];  // per (partial p, expert e): rows of e in earlier blocks
  __shared__ int32_t s_total[kRouteThreads];  // per (p, e): rows of e in all blocks
  __shared__ int32_t s_base[kMaxExperts];
  __shared__ int32_t s_cnt[kMaxExperts];
  __shared__ int32_t s_off[kMaxExperts + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int E = a.E, k = a.k, b = blockIdx.x;

  // thread (p, e) sums histogram rows [b0, b1) of column e, kHistLoads loads in flight
  const int P = kRouteThreads / E;  // partial sums per expert (>= 2)
  const int chunk = (nblk + P - 1) / P;
  const int e = threadIdx.x % E, p = threadIdx.x / E;
  if (p < P) {
    const int b0 = p * chunk, b1 = min(nblk, b0 + chunk);
    int below = 0, total = 0;
    for (int bb = b0; bb < b1; bb += kHistLoads) {
      int hv[kHistLoads];
#pragma unroll
      for (int u = 0; u < kHistLoads; ++u)
        hv[u] = bb + u < b1 ? __ldg(a.hist + static_cast<size_t>(bb + u) * E + e) : 0;
#pragma unroll
      for (int u = 0; u < kHistLoads; ++u) {
        total += hv[u];
        below += bb + u < b ? hv[u] : 0;
      }
    }
    s_below[p * E + e] = below;
    s_total[p * E + e] = total;
  }
  __syncthreads();
  if (threadIdx.x < E) {
    int below = 0, total = 0;
    for (int q = 0; q < P; ++q) {
      below += s_below[q * E + threadIdx.x];
      total += s_total[q * E + threadIdx.x];
    }
    s_base[threadIdx.x] = below;
    s_cnt[threadIdx.x] = total;
    if (b == 0) a.counts[threadIdx.x] = total;
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
  if (b == 0 && threadIdx.x <= E) a.offsets[threadIdx.x] = s_off[threadIdx.x];

  // this block's slots: row = start of expert e + rows of e in earlier blocks + rank
  const int t0 = b * TB, ntok = min(TB, a.T - t0);
  for (int sl = threadIdx.x; sl < ntok * k; sl += kRouteThreads) {
    const size_t s = static_cast<size_t>(t0) * k + sl;
    const int ee = a.topk_idx[s];
    const int row = s_off[ee] + s_base[ee] + a.lrank[s];
    a.row_of_slot[s] = row;
    a.slot_of_row[row] = static_cast<int32_t>(s);
    a.w_row[row] = a.topk_w[s];
  }
}

}  // namespace

int route_num_blocks(int T) { return (T + TB - 1) / TB; }

template <int KMAX>
cudaError_t launch_topk(const RouteArgs &a, cudaStream_t s) {
  const int nblk = route_num_blocks(a.T);
  const size_t smem = static_cast<size_t>(TB) * logit_stride(a.E) * sizeof(float);
  static DeviceOnce once;  // the shared-memory opt-in (room for E = 256), once per device
  const cudaError_t e = once.get([](int *) {
    return cudaFuncSetAttribute(route_topk_kernel<KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TB * logit_stride(kMaxExperts) * static_cast<int>(sizeof(float)));
  });
  if (e != cudaSuccess) return e;
  route_topk_kernel<KMAX><<<nblk, kRouteThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_route_topk(const RouteArgs &a, cudaStream_t s) {
  return a.k <= 8 ? launch_topk<8>(a, s) : launch_topk<kMaxTopK>(a, s);
}

cudaError_t launch_route_index(const RouteArgs &a, cudaStream_t s) {
  const int nblk = route_num_blocks(a.T);
  route_index_kernel<<<nblk, kRouteThreads, 0, s>>>(a, nblk);
  return cudaGetLastError();
}

}  // namespace moe
