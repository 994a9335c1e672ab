// gather.cu -- the memory-bound row movements of the layer.
//
// On one GPU the expert-parallel exchange of the pages (dispatch: tokens are
// permuted and sent to their experts; combine: results come back and are
// accumulated in token order -- NVIDIA MoE article, "Optimizacion 2") becomes
// a device-memory permute and a gather-sum.  All kernels use one warp per
// token and 16-byte vectors; every token row is read once, every permuted row
// written once.  Sums run over the token's k choices in a fixed order (j =
// 0..k-1) in fp32, so results are deterministic (no atomics).
//
//   permute_rows : x_perm[row(t,j)] = x[t]                      (dispatch)
//   gather_sum   : out[t] = sum_j w_tj * Y[row(t,j)]           (combine)
//                  dx[t]  = sum_j dX_perm[row(t,j)]            (un-permute)
//   router_grad  : from g_tj = <dy[t], Y[row(t,j)]> (d w_tj) in partial sums
//                  per permuted row: d_topk_w and
//                  d_logits[t, S_tj] = w_tj (g_tj - sum_i w_ti g_ti), 0 elsewhere
#include "common.cuh"
#include "mxfp8.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;       // warps (tokens) per block
constexpr int kVecPerLane = 8;  // 16-byte vectors per lane per chunk: 2048 bf16 per warp

__device__ __forceinline__ void accum8(float (&acc)[8], const uint4 &q, float w) {
  acc[0] = fmaf(w, bf16_lo(q.x), acc[0]);
  acc[1] = fmaf(w, bf16_hi(q.x), acc[1]);
  acc[2] = fmaf(w, bf16_lo(q.y), acc[2]);
  acc[3] = fmaf(w, bf16_hi(q.y), acc[3]);
  acc[4] = fmaf(w, bf16_lo(q.z), acc[4]);
  acc[5] = fmaf(w, bf16_hi(q.z), acc[5]);
  acc[6] = fmaf(w, bf16_lo(q.w), acc[6]);
  acc[7] = fmaf(w, bf16_hi(q.w), acc[7]);
}

__device__ __forceinline__ float dot8(const uint4 &a, const uint4 &b) {
  float s = bf16_lo(a.x) * bf16_lo(b.x);
  s = fmaf(bf16_hi(a.x), bf16_hi(b.x), s);
  s = fmaf(bf16_lo(a.y), bf16_lo(b.y), s);
  s = fmaf(bf16_hi(a.y), bf16_hi(b.y), s);
  s = fmaf(bf16_lo(a.z), bf16_lo(b.z), s);
  s = fmaf(bf16_hi(a.z), bf16_hi(b.z), s);
  s = fmaf(bf16_lo(a.w), bf16_lo(b.w), s);
  s = fmaf(bf16_hi(a.w), bf16_hi(b.w), s);
  return s;
}

__global__ void __launch_bounds__(kWarps * 32) permute_rows_kernel(const uint4 *__restrict__ x,
                                                                  const int32_t *__restrict__ ros,
                                                                  uint4 *__restrict__ xp, int T,
                                                                  int nv, int k) {
  griddep_wait();  // the previous kernel in the stream has completed
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const int myrow = lane < k ? __ldg(ros + static_cast<size_t>(t) * k + lane) : 0;
  for (int v0 = 0; v0 < nv; v0 += 32 * kVecPerLane) {
    uint4 buf[kVecPerLane];
#pragma unroll
    for (int u = 0; u < kVecPerLane; ++u) {
      const int v = v0 + u * 32 + lane;
      if (v < nv) buf[u] = __ldcs(x + static_cast<size_t>(t) * nv + v);
    }
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, myrow, j);
      uint4 *dst = xp + static_cast<size_t>(row) * nv;
#pragma unroll
      for (int u = 0; u < kVecPerLane; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < nv) dst[v] = buf[u];
      }
    }
  }
}

// The mxfp8 forward's dispatch: each token's row quantised along H once (a
// 32-element block is four consecutive 16-byte vectors, i.e. four neighbouring
// lanes) with its codes and scale written to the padded row of each of its k
// permuted rows (expert e's rows start at pad_off[e]); x_perm as above only
// when xp is set (the mxfp8 GEMMs read the codes, and its backward gathers x).
__global__ void __launch_bounds__(kWarps * 32) permute_quant_kernel(
    const uint4 *__restrict__ x, const int32_t *__restrict__ ros, const int32_t *__restrict__ topk_idx,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ pad_off, uint4 *__restrict__ xp,
    uint8_t *__restrict__ codes, uint8_t *__restrict__ sf, SfLayout L, int T, int nv, int k) {
  griddep_wait();  // the previous kernel in the stream has completed
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const int H = nv * 8;
  int myrow = 0, myprow = 0;
  if (lane < k) {
    myrow = __ldg(ros + static_cast<size_t>(t) * k + lane);
    const int e = __ldg(topk_idx + static_cast<size_t>(t) * k + lane);
    myprow = __ldg(pad_off + e) + myrow - __ldg(offsets + e);
  }
  for (int v0 = 0; v0 < nv; v0 += 32 * kVecPerLane) {
    uint4 buf[kVecPerLane];
    uint2 q[kVecPerLane];
    uint32_t sfw[kVecPerLane];
#pragma unroll
    for (int u = 0; u < kVecPerLane; ++u) {
      const int v = v0 + u * 32 + lane;
      buf[u] = v < nv ? __ldcs(x + static_cast<size_t>(t) * nv + v) : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {buf[u].x, buf[u].y, buf[u].z, buf[u].w};
      float f[8];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        f[2 * h] = bf16_lo(w[h]);
        f[2 * h + 1] = bf16_hi(w[h]);
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // the block's four lanes
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const int X = mx_scale_exp(amax);
      const float s = pow2_neg(X);
      q[u] = make_uint2(pack_e4m3x4_scaled(f[0], f[1], f[2], f[3], s),
                        pack_e4m3x4_scaled(f[4], f[5], f[6], f[7], s));
      // the four scale codes of K blocks (v >> 2) .. + 3, one atom word, gathered in
      // lanes 0 and 16 (K blocks 8u + 4 (lane / 16) ..; H % 128 == 0, so a word is
      // whole when its first block is inside the row)
      const uint32_t c = static_cast<uint32_t>(X + 127);
      sfw[u] = c | (__shfl_down_sync(0xffffffffu, c, 4) << 8) | (__shfl_down_sync(0xffffffffu, c, 8) << 16) |
               (__shfl_down_sync(0xffffffffu, c, 12) << 24);
    }
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, myrow, j);
      const int prow = __shfl_sync(0xffffffffu, myprow, j);
      uint4 *dst = xp + static_cast<size_t>(row) * nv;
      uint2 *cdst = reinterpret_cast<uint2 *>(codes + static_cast<size_t>(prow) * H);
      uint8_t *rsf = sf + atom_row_sg<128>(0, prow, H, L.seg);  // one segment, groups of 128
#pragma unroll
      for (int u = 0; u < kVecPerLane; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < nv) {
          if (xp) dst[v] = buf[u];
          cdst[v] = q[u];
          if ((lane & 15) == 0) *reinterpret_cast<uint32_t *>(rsf + atom_kblock(v >> 2)) = sfw[u];
        }
      }
    }
  }
}

// Padded rows past each expert's count (up to the next 128-row boundary): zero
// codes and zero scale codes.  One block per expert, a warp per row: 16-byte
// pieces of codes, and the row's scale words (four K blocks each) at the row's
// atom position (scales in one segment, groups of 128 rows).
__global__ void __launch_bounds__(256) zero_pad_rows_kernel(const int32_t *__restrict__ offsets,
                                                            const int32_t *__restrict__ pad_off, int K,
                                                            uint8_t *__restrict__ codes,
                                                            uint8_t *__restrict__ sf, int seg) {
  griddep_wait();  // the previous kernel in the stream has completed
  const int e = blockIdx.x, lane = threadIdx.x & 31;
  const int first = __ldg(pad_off + e) + (__ldg(offsets + e + 1) - __ldg(offsets + e));
  const int end = __ldg(pad_off + e + 1);
  for (int r = first + (threadIdx.x >> 5); r < end; r += blockDim.x >> 5) {
    uint4 *row = reinterpret_cast<uint4 *>(codes + static_cast<size_t>(r) * K);
    for (int c = lane; c < K / 16; c += 32) row[c] = make_uint4(0, 0, 0, 0);
    uint8_t *rsf = sf + atom_row_sg<128>(0, r, K, seg);
    for (int j = lane; j < K / 128; j += 32) *reinterpret_cast<uint32_t *>(rsf + static_cast<size_t>(j) * 512) = 0u;
  }
}

template <bool kWeighted>
__global__ void __launch_bounds__(kWarps * 32) gather_sum_kernel(const uint4 *__restrict__ rows,
                                                                const int32_t *__restrict__ ros,
                                                                const float *__restrict__ w,
                                                                uint4 *__restrict__ out, int T,
                                                                int nv, int k) {
  griddep_wait();  // the previous kernel in the stream has completed
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const int myrow = lane < k ? __ldg(ros + static_cast<size_t>(t) * k + lane) : 0;
  const float myw = (kWeighted && lane < k) ? __ldg(w + static_cast<size_t>(t) * k + lane) : 1.f;
  for (int v0 = 0; v0 < nv; v0 += 32 * kVecPerLane) {
    float acc[kVecPerLane][8];
#pragma unroll
    for (int u = 0; u < kVecPerLane; ++u)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[u][c] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, myrow, j);
      const float wj = __shfl_sync(0xffffffffu, myw, j);
      const uint4 *src = rows + static_cast<size_t>(row) * nv;
      uint4 q[kVecPerLane];
#pragma unroll
      for (int u = 0; u < kVecPerLane; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < nv) q[u] = __ldcs(src + v);
      }
#pragma unroll
      for (int u = 0; u < kVecPerLane; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < nv) accum8(acc[u], q[u], wj);
      }
    }
#pragma unroll
    for (int u = 0; u < kVecPerLane; ++u) {
      const int v = v0 + u * 32 + lane;
      if (v < nv) {
        uint4 r;
        r.x = pack_bf16x2(acc[u][0], acc[u][1]);
        r.y = pack_bf16x2(acc[u][2], acc[u][3]);
        r.z = pack_bf16x2(acc[u][4], acc[u][5]);
        r.w = pack_bf16x2(acc[u][6], acc[u][7]);
        out[static_cast<size_t>(t) * nv + v] = r;
      }
    }
  }
}

// Router gradients of token t from g_tj (lane j < k holds g, w, expert of
// choice j): d_topk_w = g, and d_logits[t, S_tj] = w_j (g_j - sum_i w_i g_i),
// written as w_j sum_i w_i (g_j - g_i) (the weights sum to one): no
// cancellation when one weight is close to 1; zero for the other experts.
__device__ __forceinline__ void router_grads(float myg, float myw, int mye, size_t t, int k, int E,
                                             float *__restrict__ d_logits, float *__restrict__ d_topk_w) {
  const int lane = threadIdx.x & 31;
  if (d_topk_w && lane < k) d_topk_w[t * k + lane] = myg;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxTopK; ++i)
    if (i < k) acc = fmaf(__shfl_sync(0xffffffffu, myw, i), myg - __shfl_sync(0xffffffffu, myg, i), acc);
  const float mydl = myw * acc;
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int e = e0 + lane;
    float val = 0.f;
    for (int j = 0; j < k; ++j) {
      const int ej = __shfl_sync(0xffffffffu, mye, j);
      const float dj = __shfl_sync(0xffffffffu, mydl, j);
      if (ej == e) val = dj;
    }
    if (e < E) d_logits[t * E + e] = val;
  }
}

// d_logits and d_topk_w of a token from g_tj in np partial sums per permuted
// row (the bf16 dA GEMM's epilogue: g_tj = <dy_t . W_down^T, A_r>; the fp8
// modes' pass over dy: <dy_t, Y_r>), added here for row r = row(t,j) in a fixed
// order.
__global__ void __launch_bounds__(kWarps * 32) router_grad_kernel(
    const int32_t *__restrict__ ros, const int32_t *__restrict__ topk_idx, const float *__restrict__ topk_w,
    const float *__restrict__ g_part, int np, float *__restrict__ d_logits, float *__restrict__ d_topk_w,
    int T, int E, int k) {
  griddep_wait();  // the previous kernel in the stream has completed
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const size_t sb = static_cast<size_t>(t) * k;
  float myg = 0.f, myw = 0.f;
  int mye = -1;
  if (lane < k) {
    const float *gp = g_part + static_cast<size_t>(__ldg(ros + sb + lane)) * np;
    for (int p = 0; p < np; ++p) myg += __ldg(gp + p);
    myw = __ldg(topk_w + sb + lane);
    mye = __ldg(topk_idx + sb + lane);
  }
  router_grads(myg, myw, mye, static_cast<size_t>(t), k, E, d_logits, d_topk_w);
}

inline int blocks_for(int T) { return (T + kWarps - 1) / kWarps; }

}  // namespace

cudaError_t launch_permute_rows(const uint16_t *x, const int32_t *row_of_slot, uint16_t *x_perm,
                                int T, int H, int k, cudaStream_t s) {
  return launch_pdl(permute_rows_kernel, dim3(blocks_for(T)), dim3(kWarps * 32), 0, s, 1,
                    reinterpret_cast<const uint4 *>(x), row_of_slot, reinterpret_cast<uint4 *>(x_perm), T, H / 8,
                    k);
}

cudaError_t launch_gather_sum(const uint16_t *rows, const int32_t *row_of_slot, const float *w,
                              uint16_t *out, int T, int H, int k, cudaStream_t s) {
  return launch_pdl(w ? gather_sum_kernel<true> : gather_sum_kernel<false>, dim3(blocks_for(T)),
                    dim3(kWarps * 32), 0, s, 1, reinterpret_cast<const uint4 *>(rows), row_of_slot, w,
                    reinterpret_cast<uint4 *>(out), T, H / 8, k);
}

namespace {

// Router projection backward: d_logits rounded to bf16 (nearest even) for the
// two bf16 tensor-core products, four floats per thread; the first block also
// writes the weight gradient's S token segments (S + 1 offsets, segment i =
// tokens [T i / S, T (i+1) / S)).
__global__ void __launch_bounds__(256) router_dlogits_kernel(const float4 *__restrict__ in, uint2 *__restrict__ out,
                                                             int64_t n4, int32_t *split, int T, int S) {
  griddep_wait();  // the previous kernel in the stream has completed
  if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) <= S)
    split[threadIdx.x] = static_cast<int32_t>(static_cast<int64_t>(T) * threadIdx.x / S);
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 v = __ldg(in + i);
  out[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

// out[i] = sum over s of parts[s][i], s ascending (a fixed order: deterministic).
__global__ void __launch_bounds__(256) sum_segments_kernel(const float4 *__restrict__ parts, int S, int64_t n4,
                                                           float4 *__restrict__ out) {
  griddep_wait();  // the previous kernel in the stream has completed
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  float4 a = __ldg(parts + i);
  for (int s = 1; s < S; ++s) {
    const float4 b = __ldg(parts + static_cast<int64_t>(s) * n4 + i);
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
  }
  out[i] = a;
}

}  // namespace

cudaError_t launch_router_dlogits(const float *d_logits, uint16_t *out, int64_t n, int32_t *split, int T, int S,
                                  cudaStream_t s) {
  if (S < 1 || S > 63) return cudaErrorInvalidValue;
  const int64_t n4 = n / 4;  // n = T * E, a multiple of 8 (E % 8 == 0)
  const int64_t blocks = (n4 + 255) / 256;
  return launch_pdl(router_dlogits_kernel, dim3(static_cast<unsigned>(blocks > 0 ? blocks : 1)), dim3(256), 0, s,
                    1, reinterpret_cast<const float4 *>(d_logits), reinterpret_cast<uint2 *>(out), n4, split, T, S);
}

cudaError_t launch_sum_segments(const float *parts, int S, int64_t n, float *out, cudaStream_t s) {
  const int64_t n4 = n / 4;  // n = H * E, a multiple of 8
  if (n4 == 0) return cudaSuccess;
  return launch_pdl(sum_segments_kernel, dim3(static_cast<unsigned>((n4 + 255) / 256)), dim3(256), 0, s, 1,
                    reinterpret_cast<const float4 *>(parts), S, n4, reinterpret_cast<float4 *>(out));
}

cudaError_t launch_permute_quant(const uint16_t *x, const int32_t *row_of_slot, const int32_t *topk_idx,
                                 const int32_t *offsets, const int32_t *pad_off, uint16_t *x_perm,
                                 uint8_t *codes, uint8_t *sf, SfLayout L, int T, int H, int k, cudaStream_t s) {
  if (L.group != 128 || H % 128 != 0) return cudaErrorInvalidValue;  // padded rows in one segment (L.seg)
  return launch_pdl(permute_quant_kernel, dim3(blocks_for(T)), dim3(kWarps * 32), 0, s, 1,
                    reinterpret_cast<const uint4 *>(x), row_of_slot, topk_idx, offsets, pad_off,
                    reinterpret_cast<uint4 *>(x_perm), codes, sf, L, T, H / 8, k);
}

cudaError_t launch_zero_pad_rows(const int32_t *offsets, const int32_t *pad_off, int E, int K, uint8_t *codes,
                                 uint8_t *sf, SfLayout L, cudaStream_t s) {
  if (L.group != 128 || K % 128 != 0) return cudaErrorInvalidValue;  // padded rows in one segment (L.seg)
  return launch_pdl(zero_pad_rows_kernel, dim3(E), dim3(256), 0, s, 1, offsets, pad_off, K, codes, sf, L.seg);
}

cudaError_t launch_router_grad(const int32_t *row_of_slot, const int32_t *topk_idx, const float *topk_w,
                               const float *g_part, int np, float *d_logits, float *d_topk_w, int T, int E, int k,
                               cudaStream_t s) {
  return launch_pdl(router_grad_kernel, dim3(blocks_for(T)), dim3(kWarps * 32), 0, s, 1, row_of_slot, topk_idx,
                    topk_w, g_part, np, d_logits, d_topk_w, T, E, k);
}

}  // namespace moe
