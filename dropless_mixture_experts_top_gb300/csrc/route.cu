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
//   route_topk  : the block's 64 tokens' logits staged in shared memory (all
//                 of a thread's loads issued before the first store); four
//                 threads per token, each taking every fourth expert.  Each
//                 thread keeps the KMAX/4 largest of its logits (values only,
//                 two min/max per logit); the smallest of those over the four
//                 threads is a threshold with at least KMAX >= k logits at or
//                 above it, so the top k are among them.  Only those
//                 candidates (typically a tenth of the row) enter a sorted
//                 KMAX list per thread; the four lists merge by two shuffle
//                 rounds (bitonic).  Ties -> lower expert.  fp32 renormalised
//                 weights.  Every token's chosen experts set one bit in a
//                 per-expert bitmask over the block's tokens, so a slot's rank
//                 in its (block, expert) run is a popcount (one byte per slot)
//                 and the block's histogram row the masks' popcounts.  The
//                 scan over blocks runs in the same launch without any block
//                 waiting for another: the last block of each group of 32 to
//                 finish (an atomic ticket) turns the group's histogram rows
//                 into exclusive prefixes inside the group and writes the
//                 group's totals; the last group to finish scans the group
//                 totals over groups (exclusive) and the expert totals over
//                 experts (counts, offsets).  Every histogram entry is read
//                 twice, so the scan is linear in T.
//   route_index : one thread per slot: row = offsets[e] + the prefix of its
//                 group + the prefix of its block inside the group + its rank;
//                 row_of_slot, slot_of_row, w_row.
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
constexpr int kScanGroup = 32;              // route blocks per scan group (one load each in flight)

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
// block's first token is a multiple of 64) into shared memory rows of S
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
  griddep_wait();  // the previous kernel in the stream has completed
  extern __shared__ __align__(16) float s_lg[];           // [TB][E + 4] this block's logits
  __shared__ uint32_t s_emask[kMaxExperts][kMaskWords];  // tokens of this block that chose expert e
  __shared__ uint8_t s_slot_e[TB * kMaxTopK];            // expert of each of the block's slots
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, k = a.k, T = a.T;
  const int S = logit_stride(E);
  const int b = blockIdx.x, nblk = gridDim.x;
  const int t0 = b * TB;
  const int ntok = min(TB, T - t0);

  for (int i = threadIdx.x; i < E * kMaskWords; i += kRouteThreads) (&s_emask[0][0])[i] = 0u;
  const bool bad = stage_logits(a.logits + static_cast<size_t>(t0) * E, ntok * E, E, S, s_lg);
  __syncthreads();

  // Top-k of token tl by its kQ threads (lanes kTokPerWarp apart): quarter qq
  // takes experts qq, qq + kQ, qq + 2kQ, ...
  {
    const int tl = warp * kTokPerWarp + lane % kTokPerWarp, qq = lane / kTokPerWarp;
    const int nm = tl < ntok ? (E - qq + kQ - 1) / kQ : 0;  // this quarter's experts (<= 64)
    const float *row = s_lg + tl * S;
    // the quarter's MQ largest logits, descending (-inf while it has fewer)
    constexpr int MQ = KMAX / kQ;
    float qmax[MQ];
#pragma unroll
    for (int j = 0; j < MQ; ++j) qmax[j] = -INFINITY;
    for (int m = 0; m < nm; ++m) {
      const float v = row[qq + kQ * m];
#pragma unroll
      for (int j = MQ - 1; j > 0; --j) qmax[j] = fmaxf(qmax[j], fminf(qmax[j - 1], v));
      qmax[0] = fmaxf(qmax[0], v);
    }
    // every quarter holds MQ logits >= its qmax[MQ-1] (or has fewer, and then
    // tau is -inf): at least kQ * MQ = KMAX >= k logits are >= tau, so the k-th
    // largest is too, and every logit of the top k is a candidate
    float tau = qmax[MQ - 1];
#pragma unroll
    for (int o = kTokPerWarp; o < 32; o <<= 1) tau = fminf(tau, __shfl_xor_sync(0xffffffffu, tau, o));
    uint64_t cand = 0;
    for (int m = 0; m < nm; ++m) cand |= static_cast<uint64_t>(row[qq + kQ * m] >= tau) << m;
    float tv[KMAX];
    int ti[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      tv[j] = -INFINITY;
      ti[j] = INT_MAX;
    }
    while (cand) {  // insert each candidate into the sorted list
      const int m = __ffsll(static_cast<long long>(cand)) - 1;
      cand &= cand - 1;
      const float v = row[qq + kQ * m];
      const int e = qq + kQ * m;
      // its position p = the entries that rank before it (independent compares);
      // the entries from p on move down one place and the last drops out
      int p = 0;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) p += ranks_before(tv[j], ti[j], v, e) ? 1 : 0;
#pragma unroll
      for (int j = KMAX - 1; j > 0; --j) {
        tv[j] = j > p ? tv[j - 1] : (j == p ? v : tv[j]);
        ti[j] = j > p ? ti[j - 1] : (j == p ? e : ti[j]);
      }
      tv[0] = p == 0 ? v : tv[0];
      ti[0] = p == 0 ? e : ti[0];
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
#pragma unroll
    for (int w = 0; w < kMaskWords - 1; ++w) r += w < (tl >> 5) ? __popc(mk[w]) : 0;
    a.lrank[static_cast<size_t>(t0) * k + sl] = static_cast<uint8_t>(r);
  }
  // the block's histogram row (kRouteThreads >= E)
  if (threadIdx.x < E) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < kMaskWords; ++w) c += __popc(s_emask[threadIdx.x][w]);
    a.hist[static_cast<size_t>(b) * E + threadIdx.x] = c;
  }

  // ---- scan over blocks: the last block of the group to arrive takes the group
  const int g = b / kScanGroup, ngroups = (nblk + kScanGroup - 1) / kScanGroup;
  const int gb0 = g * kScanGroup, gn = min(kScanGroup, nblk - gb0);
  // one thread per block fences and takes the ticket: the barrier orders the
  // block's writes before its fence, so they are visible before the ticket
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const bool last = atomicAdd(a.tickets + 1 + g, 1) == gn - 1;
    if (last) __threadfence();  // the group's rows, seen through the ticket, before they are read
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;
  if (threadIdx.x < E) {  // column e: exclusive prefix of the group's rows, in place; the group total
    const int e = threadIdx.x;
    int h[kScanGroup];
#pragma unroll
    for (int i = 0; i < kScanGroup; ++i)
      h[i] = i < gn ? __ldcg(a.hist + static_cast<size_t>(gb0 + i) * E + e) : 0;
    int run = 0;
#pragma unroll
    for (int i = 0; i < kScanGroup; ++i) {
      if (i < gn) a.hist[static_cast<size_t>(gb0 + i) * E + e] = run;
      run += h[i];
    }
    a.gpref[static_cast<size_t>(g) * E + e] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const bool last = atomicAdd(a.tickets, 1) == ngroups - 1;
    if (last) __threadfence();
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;
  // the last group: exclusive prefix of the group totals over groups (in place),
  // expert totals (counts), and their exclusive scan over experts (offsets)
  __shared__ int32_t s_cnt[kMaxExperts];
  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    int run = 0;
    for (int g0 = 0; g0 < ngroups; g0 += kScanGroup) {
      int h[kScanGroup];
#pragma unroll
      for (int i = 0; i < kScanGroup; ++i)
        h[i] = g0 + i < ngroups ? __ldcg(a.gpref + static_cast<size_t>(g0 + i) * E + e) : 0;
#pragma unroll
      for (int i = 0; i < kScanGroup; ++i) {
        if (g0 + i < ngroups) a.gpref[static_cast<size_t>(g0 + i) * E + e] = run;
        run += h[i];
      }
    }
    s_cnt[e] = run;
    a.counts[e] = run;
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
      if (ee < E) a.offsets[ee] = carry + incl - c;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) a.offsets[E] = carry;
  }
}

__global__ void __launch_bounds__(256) route_index_kernel(RouteArgs a) {
  griddep_wait();  // the previous kernel in the stream has completed
  const int s = blockIdx.x * 256 + threadIdx.x;  // slot t * k + j
  if (s >= a.T * a.k) return;
  const int e = __ldg(a.topk_idx + s), r = __ldg(a.lrank + s);
  const float w = __ldg(a.topk_w + s);
  const int b = s / a.k / TB, E = a.E;
  const int row = __ldg(a.offsets + e) + __ldg(a.gpref + static_cast<size_t>(b / kScanGroup) * E + e) +
                  __ldg(a.hist + static_cast<size_t>(b) * E + e) + r;
  a.row_of_slot[s] = row;
  a.slot_of_row[row] = s;
  a.w_row[row] = w;
}

}  // namespace

int route_num_blocks(int T) { return (T + TB - 1) / TB; }
int route_scan_groups(int T) { return (route_num_blocks(T) + kScanGroup - 1) / kScanGroup; }

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
  return launch_pdl(route_topk_kernel<KMAX>, dim3(nblk), dim3(kRouteThreads), smem, s, 1, a);
}

cudaError_t launch_route_topk(const RouteArgs &a, cudaStream_t s) {
  return a.k <= 8 ? launch_topk<8>(a, s) : launch_topk<kMaxTopK>(a, s);
}

cudaError_t launch_route_index(const RouteArgs &a, cudaStream_t s) {
  const int slots = a.T * a.k;
  return launch_pdl(route_index_kernel, dim3((slots + 255) / 256), dim3(256), 0, s, 1, a);
}

}  // namespace moe
