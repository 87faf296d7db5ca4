// fathom_sparse_attn: exact attention over the k selected keys of each row,
// with the original (16-bit or fp32) K/V rows (Fathom article, "What the model
// keeps in memory": compare the query with the keys and mix the values by
// relevance; "The first fix": attend over just the k winners).  Every query
// head of a KV head uses its own q with that KV head's winner set.
//
// GPU form: one thread-block cluster of 16 (or the portable 8) CTAs per KV head.  Each CTA
// takes a slice of the winners; each warp gathers whole K and V rows (a lane
// holds 4 channels: 8 contiguous bytes of a 16-bit row), several winners in
// flight per warp, reduces the group's dot products with shuffles and keeps an
// online softmax (running max, sum and weighted V).  The CTA merges its warps
// in shared memory; then CTA 0 of the cluster merges the cluster's partials by
// reading the other CTAs' shared memory (distributed shared memory) and writes
// the output: one launch, no partials in global memory.  The K/V rows may sit
// in HBM or in pinned host memory.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace fathom {
namespace {

constexpr int kClusterMax = 16;  // CTAs per KV head when non-portable clusters are allowed, else 8
constexpr int kUnroll = 4;       // winners in flight per warp

// threads per CTA: 512 while the per-thread state (G heads) stays small, else 256
template <int G>
constexpr int attn_threads() { return G <= 4 ? 512 : 256; }

template <typename T>
struct Row4;
template <>
struct Row4<float> {
  __device__ static float4 get(const float* p, int64_t row, int64_t stride, int lane) {
    return __ldg(reinterpret_cast<const float4*>(p + row * stride) + lane);
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

// weight of a partial with running max mw when merged under the overall max M
__device__ __forceinline__ float merge_weight(float mw, float M) { return mw == -INFINITY ? 0.0f : expf(mw - M); }

template <int G, typename KV, int T = attn_threads<G>()>
__global__ void __launch_bounds__(T) attn_cluster_kernel(int64_t n, int64_t k, int64_t stride,
                                                                    const void* __restrict__ q, int q_dtype,
                                                                    const KV* __restrict__ K, const KV* __restrict__ V,
                                                                    const int32_t* __restrict__ idx,
                                                                    float* __restrict__ out,
                                                                    uint16_t* __restrict__ out_bf16) {
  __shared__ float s_q[G][kD];
  constexpr int kWarps = T / 32;
  __shared__ float s_m[kWarps][G], s_l[kWarps][G];
  __shared__ float s_o[kWarps][G][kD];
  __shared__ float c_m[G], c_l[G];  // this CTA's merged partial, read by CTA 0 of the cluster
  __shared__ float c_o[G][kD];
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = int(cluster.block_rank());
  const int csize = int(cluster.num_blocks());
  const int r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float scale = 0.08838834764831845f;  // 1/sqrt(128)
  for (int i = tid; i < G * kD; i += T)
    s_q[i / kD][i % kD] = load_as_float(q, int64_t(r) * G * kD + i, q_dtype) * scale;
  __syncthreads();
  float4 qv[G];
#pragma unroll
  for (int h = 0; h < G; ++h)
    qv[h] = make_float4(s_q[h][4 * lane], s_q[h][4 * lane + 1], s_q[h][4 * lane + 2], s_q[h][4 * lane + 3]);
  const int64_t per = (k + csize - 1) / csize;
  const int64_t i0 = int64_t(crank) * per, i1 = (i0 + per < k) ? i0 + per : k;
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
  for (int64_t base = i0 + int64_t(warp) * kUnroll; base < i1; base += int64_t(kWarps) * kUnroll) {
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
        const float corr = expf(m[h] - mn);  // m = -inf the first time: exp(-inf) = 0
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
  // merge the warps of this CTA
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
  for (int e = tid; e < G * kD; e += T) {
    const int h = e / kD, c = e % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][h]);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float wt = merge_weight(s_m[w][h], M);
      L = fmaf(s_l[w][h], wt, L);
      O = fmaf(s_o[w][h][c], wt, O);
    }
    c_o[h][c] = O;
    if (c == 0) {
      c_m[h] = M;
      c_l[h] = L;
    }
  }
  cluster.sync();  // every CTA's partial is visible to the cluster
  if (crank == 0) {
    for (int e = tid; e < G * kD; e += T) {
      const int h = e / kD, c = e % kD;
      float M = -INFINITY;
      for (int rk = 0; rk < csize; ++rk) M = fmaxf(M, *cluster.map_shared_rank(&c_m[h], rk));
      float L = 0.0f, O = 0.0f;
      for (int rk = 0; rk < csize; ++rk) {
        const float wt = merge_weight(*cluster.map_shared_rank(&c_m[h], rk), M);
        L = fmaf(*cluster.map_shared_rank(&c_l[h], rk), wt, L);
        O = fmaf(*cluster.map_shared_rank(&c_o[h][c], rk), wt, O);
      }
      const float v = L > 0.0f ? O / L : 0.0f;
      const int64_t qh = int64_t(r) * G + h;
      if (out) out[qh * kD + c] = v;
      if (out_bf16) {
        const __nv_bfloat16 b = __float2bfloat16_rn(v);
        out_bf16[qh * kD + c] = *reinterpret_cast<const uint16_t*>(&b);
      }
    }
  }
  cluster.sync();  // keep this CTA's shared memory alive until CTA 0 has read it
}

template <int G, typename KV>
cudaError_t launch_attn_t(int rows, int64_t n, int64_t k, const void* q, int q_dtype, const void* K, const void* V,
                          int64_t stride, const int32_t* idx, float* out, uint16_t* out_bf16, cudaStream_t st) {
  auto kern = attn_cluster_kernel<G, KV>;
  // 16-CTA clusters need an opt-in per kernel; fall back to the portable 8 if it is refused
  static int cluster = 0;
  if (cluster == 0) {
    cluster = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess
                  ? kClusterMax
                  : 8;
    cudaGetLastError();
  }
  for (;;) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(cluster), unsigned(rows), 1);
    cfg.blockDim = dim3(attn_threads<G>(), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, n, k, stride, q, q_dtype, reinterpret_cast<const KV*>(K),
                                             reinterpret_cast<const KV*>(V), idx, out, out_bf16);
    if (e == cudaSuccess || cluster == 8) return e;
    cudaGetLastError();  // the larger cluster could not be scheduled: use the portable size from now on
    cluster = 8;
  }
}

template <int G>
cudaError_t launch_attn_g(int rows, int64_t n, int64_t k, const void* q, int q_dtype, const void* K, const void* V,
                          int kv_dtype, int64_t stride, const int32_t* idx, float* out, uint16_t* out_bf16,
                          cudaStream_t st) {
  if (kv_dtype == FATHOM_F32)
    return launch_attn_t<G, float>(rows, n, k, q, q_dtype, K, V, stride, idx, out, out_bf16, st);
  if (kv_dtype == FATHOM_F16)
    return launch_attn_t<G, __half>(rows, n, k, q, q_dtype, K, V, stride, idx, out, out_bf16, st);
  return launch_attn_t<G, __nv_bfloat16>(rows, n, k, q, q_dtype, K, V, stride, idx, out, out_bf16, st);
}

}  // namespace

size_t attn_ws_bytes(int, int, int64_t) { return 256; }

cudaError_t launch_attn(int rows, int group, int64_t n, int64_t k, const void* q, int q_dtype, const void* K,
                        const void* V, int kv_dtype, int64_t kv_stride, const int32_t* idx, float* out,
                        uint16_t* out_bf16, void* /*ws*/, cudaStream_t st) {
  switch (group) {
    case 1: return launch_attn_g<1>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, st);
    case 2: return launch_attn_g<2>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, st);
    case 3: return launch_attn_g<3>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, st);
    case 4: return launch_attn_g<4>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, st);
    case 5: return launch_attn_g<5>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, st);
    case 6: return launch_attn_g<6>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, st);
    case 7: return launch_attn_g<7>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, st);
    case 8: return launch_attn_g<8>(rows, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, st);
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
  FATHOM_TRY(device_view(workspace, "workspace", &dW, true));
  if (!dO && !dB) return set_error(FATHOM_EINVAL, "out and out_bf16 are both NULL");
  (void)ws_bytes;  // the clustered kernel keeps its partials on chip
  const size_t al = kv_dtype == FATHOM_F32 ? 16 : 8;
  if ((reinterpret_cast<uintptr_t>(dK) % al) || (reinterpret_cast<uintptr_t>(dV) % al))
    return set_error(FATHOM_EINVAL, "K and V must be %zu-byte aligned", al);
  FATHOM_TRY_CUDA(launch_attn(rows, group, n, k, dq, q_dtype, dK, dV, kv_dtype, kv_stride, (const int32_t*)dI,
                              (float*)dO, (uint16_t*)dB, const_cast<void*>(dW), as_stream(stream)));
  return FATHOM_OK;
}

}  // extern "C"
