// fathom_sparse_attn: exact attention over the k selected keys of each row,
// with the original (16-bit or fp32) K/V rows (Fathom article, "What the model
// keeps in memory": compare the query with the keys and mix the values by
// relevance; "The first fix": attend over just the k winners).  Every query
// head of a KV head uses its own q with that KV head's winner set.
//
// GPU form: the winners of a row are split across CTAs (split count sized so
// the grid covers the SMs); each warp gathers whole K and V rows (a lane holds
// 4 channels: 8 contiguous bytes of a 16-bit row), reduces the G dot products
// with shuffles and keeps an online softmax (running max, sum, weighted V);
// the CTA merges its warps and writes one partial per (row, split, head).  A
// second kernel merges the splits with the usual max-rescaled sums.  The rows
// may sit in HBM or in pinned host memory (read over the host link).
#include "common.cuh"

namespace fathom {
namespace {

constexpr int kAttnThreads = 128;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kUnroll = 4;      // winners in flight per warp
constexpr int kPartStride = kD + 2;  // m, l, o[128]
constexpr int kMinPerSplit = 32;

template <typename T>
struct Row4;
template <>
struct Row4<float> {
  using raw = float4;
  __device__ static float4 get(const float* p, int64_t row, int64_t stride, int lane) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p + row * stride) + lane);
    return v;
  }
};
template <>
struct Row4<__half> {
  __device__ static float4 get(const __half* p, int64_t row, int64_t stride, int lane) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p + row * stride) + lane);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
};
template <>
struct Row4<__nv_bfloat16> {
  __device__ static float4 get(const __nv_bfloat16* p, int64_t row, int64_t stride, int lane) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p + row * stride) + lane);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
};

template <int G, typename KV>
__global__ void __launch_bounds__(kAttnThreads) attn_partial_kernel(int64_t n, int64_t k, int64_t stride, int splits,
                                                                    const void* __restrict__ q, int q_dtype,
                                                                    const KV* __restrict__ K, const KV* __restrict__ V,
                                                                    const int32_t* __restrict__ idx,
                                                                    float* __restrict__ part) {
  __shared__ float s_q[G][kD];
  __shared__ float s_m[kAttnWarps][G], s_l[kAttnWarps][G];
  __shared__ float s_o[kAttnWarps][G][kD];
  const int r = blockIdx.y, sp = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float scale = 0.08838834764831845f;  // 1/sqrt(128)
  for (int i = tid; i < G * kD; i += kAttnThreads)
    s_q[i / kD][i % kD] = load_as_float(q, int64_t(r) * G * kD + i, q_dtype) * scale;
  __syncthreads();
  float4 qv[G];
#pragma unroll
  for (int h = 0; h < G; ++h) qv[h] = make_float4(s_q[h][4 * lane], s_q[h][4 * lane + 1], s_q[h][4 * lane + 2],
                                                 s_q[h][4 * lane + 3]);
  const int64_t per = (k + splits - 1) / splits;
  const int64_t i0 = int64_t(sp) * per, i1 = (i0 + per < k) ? i0 + per : k;
  const int32_t* ir = idx + int64_t(r) * k;
  const KV* Kr = K + int64_t(r) * n * stride;
  const KV* Vr = V + int64_t(r) * n * stride;

  float m[G], l[G];
  float4 o[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
    o[h] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int64_t base = i0 + int64_t(warp) * kUnroll; base < i1; base += int64_t(kAttnWarps) * kUnroll) {
    int32_t t[kUnroll];
    float4 kr[kUnroll], vr[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = base + u;
      t[u] = (i < i1) ? __ldg(ir + i) : -1;
      if (t[u] >= n) t[u] = -1;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (t[u] >= 0) {
        kr[u] = Row4<KV>::get(Kr, t[u], stride, lane);
        vr[u] = Row4<KV>::get(Vr, t[u], stride, lane);
      } else {
        kr[u] = vr[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (t[u] < 0) continue;  // uniform across the warp
      float z[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float d = qv[h].x * kr[u].x;
        d = fmaf(qv[h].y, kr[u].y, d);
        d = fmaf(qv[h].z, kr[u].z, d);
        d = fmaf(qv[h].w, kr[u].w, d);
        z[h] = d;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int h = 0; h < G; ++h) z[h] += __shfl_xor_sync(0xffffffffu, z[h], off);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mn = fmaxf(m[h], z[h]);
        const float corr = expf(m[h] - mn);  // m = -inf first time: exp(-inf) = 0
        const float p = expf(z[h] - mn);
        l[h] = fmaf(l[h], corr, p);
        o[h].x = fmaf(o[h].x, corr, p * vr[u].x);
        o[h].y = fmaf(o[h].y, corr, p * vr[u].y);
        o[h].z = fmaf(o[h].z, corr, p * vr[u].z);
        o[h].w = fmaf(o[h].w, corr, p * vr[u].w);
        m[h] = mn;
      }
    }
  }
  // merge the warps
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (lane == 0) {
      s_m[warp][h] = m[h];
      s_l[warp][h] = l[h];
    }
    s_o[warp][h][4 * lane] = o[h].x;
    s_o[warp][h][4 * lane + 1] = o[h].y;
    s_o[warp][h][4 * lane + 2] = o[h].z;
    s_o[warp][h][4 * lane + 3] = o[h].w;
  }
  __syncthreads();
  const int c = tid;  // kAttnThreads == kD
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, s_m[w][h]);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float e = (s_m[w][h] == -INFINITY) ? 0.0f : expf(s_m[w][h] - M);
      L = fmaf(s_l[w][h], e, L);
      O = fmaf(s_o[w][h][c], e, O);
    }
    float* pp = part + ((int64_t(r) * splits + sp) * G + h) * kPartStride;
    if (c == 0) {
      pp[0] = M;
      pp[1] = L;
    }
    pp[2 + c] = O;
  }
}

// One CTA per query head: merge the split partials.
template <int G>
__global__ void __launch_bounds__(kD) attn_combine_kernel(int splits, const float* __restrict__ part,
                                                          float* __restrict__ out, uint16_t* __restrict__ out_bf16) {
  const int qh = blockIdx.x;  // r * G + h
  const int r = qh / G, h = qh % G;
  const int c = threadIdx.x;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part[((int64_t(r) * splits + s) * G + h) * kPartStride]);
  float L = 0.0f, O = 0.0f;
  for (int s = 0; s < splits; ++s) {
    const float* pp = part + ((int64_t(r) * splits + s) * G + h) * kPartStride;
    const float e = (pp[0] == -INFINITY) ? 0.0f : expf(pp[0] - M);
    L = fmaf(pp[1], e, L);
    O = fmaf(pp[2 + c], e, O);
  }
  const float v = L > 0.0f ? O / L : 0.0f;
  if (out) out[int64_t(qh) * kD + c] = v;
  if (out_bf16) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    out_bf16[int64_t(qh) * kD + c] = *reinterpret_cast<const uint16_t*>(&b);
  }
}

int attn_splits(int rows, int64_t k) {
  const int64_t want = (2 * int64_t(num_sms()) + rows - 1) / rows;
  const int64_t maxs = (k + kMinPerSplit - 1) / kMinPerSplit;
  int64_t s = want < maxs ? want : maxs;
  return int(s < 1 ? 1 : s);
}

template <int G, typename KV>
cudaError_t launch_attn_t(int rows, int64_t n, int64_t k, const void* q, int q_dtype, const void* K, const void* V,
                          int64_t stride,
                          const int32_t* idx, float* out, uint16_t* out_bf16, float* part, cudaStream_t st) {
  const int splits = attn_splits(rows, k);
  attn_partial_kernel<G, KV><<<dim3(splits, rows), kAttnThreads, 0, st>>>(
      n, k, stride, splits, q, q_dtype, reinterpret_cast<const KV*>(K), reinterpret_cast<const KV*>(V), idx, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_combine_kernel<G><<<rows * G, kD, 0, st>>>(splits, part, out, out_bf16);
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_attn_g(int rows, int64_t n, int64_t k, const void* q, int q_dtype, const void* K, const void* V,
                          int kv_dtype, int64_t stride, const int32_t* idx, float* out, uint16_t* out_bf16, float* part,
                          cudaStream_t st) {
  if (kv_dtype == FATHOM_F32)
    return launch_attn_t<G, float>(rows, n, k, q, q_dtype, K, V, stride, idx, out, out_bf16, part, st);
  if (kv_dtype == FATHOM_F16)
    return launch_attn_t<G, __half>(rows, n, k, q, q_dtype, K, V, stride, idx, out, out_bf16, part, st);
  return launch_attn_t<G, __nv_bfloat16>(rows, n, k, q, q_dtype, K, V, stride, idx, out, out_bf16, part, st);
}

}  // namespace

size_t attn_ws_bytes(int rows, int group, int64_t k) {
  const int64_t maxs = (k + kMinPerSplit - 1) / kMinPerSplit;
  return size_t(rows) * size_t(maxs) * group * kPartStride * sizeof(float) + 256;
}

cudaError_t launch_attn(int rows, int group, int64_t n, int64_t k, const void* q, int q_dtype, const void* K,
                        const void* V, int kv_dtype, int64_t kv_stride, const int32_t* idx, float* out, uint16_t* out_bf16, void* ws,
                        cudaStream_t st) {
  float* part = reinterpret_cast<float*>(ws);
  switch (group) {
    case 1: return launch_attn_g<1>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, part, st);
    case 2: return launch_attn_g<2>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, part, st);
    case 3: return launch_attn_g<3>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, part, st);
    case 4: return launch_attn_g<4>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, part, st);
    case 5: return launch_attn_g<5>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, part, st);
    case 6: return launch_attn_g<6>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, part, st);
    case 7: return launch_attn_g<7>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, part, st);
    case 8: return launch_attn_g<8>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, part, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fathom

using namespace fathom;

extern "C" {

int fathom_sparse_attn_workspace_bytes(int rows, int group, int64_t k, size_t* bytes) {
  clear_error();
  if (rows < 1 || group < 1 || group > 8 || k < 1) return set_error(FATHOM_EINVAL, "rows, group (1..8), k out of range");
  if (!bytes) return set_error(FATHOM_EINVAL, "bytes is NULL");
  *bytes = attn_ws_bytes(rows, group, k);
  return FATHOM_OK;
}

int fathom_sparse_attn(int rows, int group, int64_t n, int64_t k, const void* q, int q_dtype, const void* K,
                       const void* V, int kv_dtype, int64_t kv_stride, const int32_t* idx, float* out,
                       uint16_t* out_bf16, void* workspace, size_t ws_bytes, void* stream) {
  clear_error();
  if (rows < 1 || rows > 65535 || group < 1 || group > 8 || n < 1 || k < 1 || n > 0x7fffffff)
    return set_error(FATHOM_EINVAL, "rows, group (1..8), n, k out of range");
  if (kv_stride < kD || (kv_stride & 3)) return set_error(FATHOM_EINVAL, "kv_stride must be >= 128, a multiple of 4");
  if (!valid_dtype(q_dtype) || !valid_dtype(kv_dtype)) return set_error(FATHOM_EINVAL, "invalid dtype");
  const void *dq, *dK, *dV, *dI, *dO, *dB, *dW;
  FATHOM_TRY(device_view(q, "q", &dq));
  FATHOM_TRY(device_view(K, "K", &dK));
  FATHOM_TRY(device_view(V, "V", &dV));
  FATHOM_TRY(device_view(idx, "idx", &dI));
  FATHOM_TRY(device_view(out, "out", &dO, true));
  FATHOM_TRY(device_view(out_bf16, "out_bf16", &dB, true));
  FATHOM_TRY(device_view(workspace, "workspace", &dW));
  if (reinterpret_cast<uintptr_t>(dW) & 255) return set_error(FATHOM_EINVAL, "workspace must be 256-byte aligned");
  if (!dO && !dB) return set_error(FATHOM_EINVAL, "out and out_bf16 are both NULL");
  if (ws_bytes < attn_ws_bytes(rows, group, k))
    return set_error(FATHOM_ENOMEM, "workspace %zu < %zu bytes", ws_bytes, attn_ws_bytes(rows, group, k));
  const size_t al = kv_dtype == FATHOM_F32 ? 16 : 8;
  if ((reinterpret_cast<uintptr_t>(dK) % al) || (reinterpret_cast<uintptr_t>(dV) % al))
    return set_error(FATHOM_EINVAL, "K and V must be %zu-byte aligned", al);
  FATHOM_TRY_CUDA(launch_attn(rows, group, n, k, dq, q_dtype, dK, dV, kv_dtype, kv_stride, (const int32_t*)dI,
                              (float*)dO,
                              (uint16_t*)dB, const_cast<void*>(dW), as_stream(stream)));
  return FATHOM_OK;
}

}  // extern "C"
