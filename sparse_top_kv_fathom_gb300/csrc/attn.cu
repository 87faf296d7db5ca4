// fathom_sparse_attn: exact attention over the k selected keys of each row,
// with the original (16-bit or fp32) K/V rows (Fathom article, "What the model
// keeps in memory": compare the query with the keys and mix the values by
// relevance; "The first fix": attend over just the k winners).  Every query
// head of a KV head uses its own q with that KV head's winner set.
//
// GPU form: one thread-block cluster of 16 (or the portable 8) CTAs per KV head.  Each CTA
// takes a slice of the winners; each warp gathers whole K and V rows (a lane
// holds 4 channels: 8 contiguous bytes of a 16-bit row) for a batch of 8
// winners at once, the indices of the next batch loaded while this one is
// reduced.  The group's dot products are reduced with shuffles and an online
// softmax (one running max per batch, sum and weighted V) is kept per head.
// The CTA merges its warps in shared memory and stores its partial into CTA 0's
// shared memory (distributed shared memory); after one cluster barrier CTA 0
// merges the cluster's partials from its own shared memory and writes the
// output: one launch, no partials in global memory.  The K/V rows may sit in
// HBM or in pinned host memory.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace fathom {
namespace {

constexpr int kClusterMax = 16;  // CTAs per KV head when non-portable clusters are allowed, else 8

// threads per CTA: 512 while the per-thread state (G heads) stays small, else 256
template <int G>
constexpr int attn_threads() { return G <= 4 ? 512 : 256; }
// winners whose K/V rows a warp has in flight at once
template <int G>
constexpr int attn_batch() { return G <= 4 ? 8 : 4; }
// heads rounded up to a power of two: value u*GP + h of a batch is (winner u, head h)
template <int G>
constexpr int attn_gp() { return G == 1 ? 1 : G == 2 ? 2 : G <= 4 ? 4 : 8; }

// Transpose-reduce of 32 values across the warp: afterwards v[0] of lane j holds
// the warp's sum of value j (31 shuffles instead of 32 x 5).
__device__ __forceinline__ float warp_transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}

// One lane's 4 channels of a K or V row, kept in the storage type until used.
template <typename T>
struct Row4;
template <>
struct Row4<float> {
  using raw = float4;
  __device__ static raw load(const float* p, int64_t row, int64_t stride, int lane) {
    return __ldg(reinterpret_cast<const float4*>(p + row * stride) + lane);
  }
  __device__ static float4 cvt(raw r) { return r; }
  __device__ static raw zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
};
template <>
struct Row4<__half> {
  using raw = uint2;
  __device__ static raw load(const __half* p, int64_t row, int64_t stride, int lane) {
    return __ldg(reinterpret_cast<const uint2*>(p + row * stride) + lane);
  }
  __device__ static float4 cvt(raw u) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  __device__ static raw zero() { return make_uint2(0u, 0u); }
};
template <>
struct Row4<__nv_bfloat16> {
  using raw = uint2;
  __device__ static raw load(const __nv_bfloat16* p, int64_t row, int64_t stride, int lane) {
    return __ldg(reinterpret_cast<const uint2*>(p + row * stride) + lane);
  }
  __device__ static float4 cvt(raw u) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  __device__ static raw zero() { return make_uint2(0u, 0u); }
};

// weight of a partial with running max mw when merged under the overall max M
__device__ __forceinline__ float merge_weight(float mw, float M) { return mw == -INFINITY ? 0.0f : expf(mw - M); }

// Shared memory of one CTA (floats): the scaled queries, the warps' partials,
// and the cluster's partials (filled in CTA 0 only, by every CTA of the cluster).
template <int G, int T>
struct AttnSmem {
  static constexpr int W = T / 32;
  static constexpr int q = 0;                              // [G][kD]
  static constexpr int wm = q + G * kD;                    // [W][G]
  static constexpr int wl = wm + W * G;                    // [W][G]
  static constexpr int wo = wl + W * G;                    // [W][G][kD]
  static constexpr int cm = wo + W * G * kD;               // [kClusterMax][G]
  static constexpr int cl = cm + kClusterMax * G;          // [kClusterMax][G]
  static constexpr int co = cl + kClusterMax * G;          // [kClusterMax][G][kD]
  static constexpr int wt = co + kClusterMax * G * kD;     // merge weights [max(W, kClusterMax)][G]
  static constexpr int mx = wt + (W > kClusterMax ? W : kClusterMax) * G;  // merged max and sum [2][G]
  static constexpr int floats = mx + 2 * G;
  static constexpr size_t bytes = size_t(floats) * sizeof(float);
};

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

template <int G, typename KV, int T = attn_threads<G>()>
__global__ void __launch_bounds__(T) attn_cluster_kernel(int64_t n, int64_t k, int64_t stride, int kv_div,
                                                         const void* __restrict__ q, int q_dtype,
                                                         const KV* __restrict__ K, const KV* __restrict__ V,
                                                         const int32_t* __restrict__ idx, float* __restrict__ out,
                                                         uint16_t* __restrict__ out_bf16) {
  using L = AttnSmem<G, T>;
  using R = Row4<KV>;
  constexpr int kWarps = T / 32;
  constexpr int U = attn_batch<G>();
  extern __shared__ float smem[];
  float* s_q = smem + L::q;
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = int(cluster.block_rank());
  const int csize = int(cluster.num_blocks());
  cluster_arrive_relaxed();  // this CTA runs; waited for before the first remote store
  const int r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per = (k + csize - 1) / csize;
  const int64_t i0 = int64_t(crank) * per, i1 = (i0 + per < k) ? i0 + per : k;
  const int32_t* ir = idx + int64_t(r) * k;
  const KV* Kr = K + int64_t(r / kv_div) * n * stride;  // kv_div > 1: row r is one query head of KV row r / kv_div
  const KV* Vr = V + int64_t(r / kv_div) * n * stride;
  constexpr int64_t kStep = int64_t(kWarps) * U;
  int64_t base = i0 + int64_t(warp) * U;
  // lane u < U holds the index of winner base + u (loaded one batch ahead)
  int32_t tl = (lane < U && base + lane < i1) ? __ldg(ir + base + lane) : -1;
  const float scale = 0.08838834764831845f;  // 1/sqrt(128)
  for (int i = tid; i < G * kD; i += T) s_q[i] = load_as_float(q, int64_t(r) * G * kD + i, q_dtype) * scale;
  __syncthreads();
  float4 qv[G];
#pragma unroll
  for (int h = 0; h < G; ++h) qv[h] = reinterpret_cast<const float4*>(s_q + h * kD)[lane];

  float m[G], l[G];
  float4 o[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
    o[h] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  constexpr int GP = attn_gp<G>();
  static_assert(U * GP <= 32, "one value per lane after the transpose-reduce");
  const int uj = lane / GP, hj = lane % GP;  // this lane's (winner, head) after the reduce
  for (; base < i1; base += kStep) {
    const int32_t tcur = tl;
    int32_t t[U];
    typename R::raw kr[U], vr[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      t[u] = __shfl_sync(0xffffffffu, tcur, u);
      if (t[u] >= n) t[u] = -1;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (t[u] >= 0) {
        kr[u] = R::load(Kr, t[u], stride, lane);
        vr[u] = R::load(Vr, t[u], stride, lane);
      } else {
        kr[u] = vr[u] = R::zero();
      }
    }
    {  // the next batch's indices travel while this batch is reduced
      const int64_t nb = base + kStep;
      tl = (lane < U && nb + lane < i1) ? __ldg(ir + nb + lane) : -1;
    }
    // partial dot products of this lane's 4 channels, value u*GP + h
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.0f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float4 kf = R::cvt(kr[u]);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float d = qv[h].x * kf.x;
        d = fmaf(qv[h].y, kf.y, d);
        d = fmaf(qv[h].z, kf.z, d);
        d = fmaf(qv[h].w, kf.w, d);
        v[u * GP + h] = d;
      }
    }
    float zj = warp_transpose_sum32(v, lane);  // logit of (winner uj, head hj)
    const int32_t tj = __shfl_sync(0xffffffffu, tcur, uj & (U - 1));
    const bool valid = uj < U && hj < G && tj >= 0 && tj < n;
    if (!valid) zj = -INFINITY;
    float mb = zj;  // max over the batch's winners, per head (lanes with equal hj)
#pragma unroll
    for (int off = GP; off < 32; off <<= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
    float mn[G], corr[G];
    float mn_own = -INFINITY;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      mn[h] = fmaxf(m[h], __shfl_sync(0xffffffffu, mb, h));
      corr[h] = mn[h] == -INFINITY ? 1.0f : __expf(m[h] - mn[h]);  // m = -inf: 0
      if (h == hj) mn_own = mn[h];
    }
    const float pj = valid ? __expf(zj - mn_own) : 0.0f;
    float ps = pj;  // sum of the batch's weights, per head
#pragma unroll
    for (int off = GP; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      l[h] = fmaf(l[h], corr[h], __shfl_sync(0xffffffffu, ps, h));
      o[h].x *= corr[h];
      o[h].y *= corr[h];
      o[h].z *= corr[h];
      o[h].w *= corr[h];
      m[h] = mn[h];
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (t[u] < 0) continue;  // warp-uniform
      const float4 vf = R::cvt(vr[u]);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float p = __shfl_sync(0xffffffffu, pj, u * GP + h);
        o[h].x = fmaf(p, vf.x, o[h].x);
        o[h].y = fmaf(p, vf.y, o[h].y);
        o[h].z = fmaf(p, vf.z, o[h].z);
        o[h].w = fmaf(p, vf.w, o[h].w);
      }
    }
  }
  // merge the warps of this CTA, then push the CTA's partial into CTA 0's slot
  float* s_m = smem + L::wm;
  float* s_l = smem + L::wl;
  float* s_o = smem + L::wo;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (lane == 0) {
      s_m[warp * G + h] = m[h];
      s_l[warp * G + h] = l[h];
    }
    reinterpret_cast<float4*>(s_o + (warp * G + h) * kD)[lane] = o[h];
  }
  float* s_wt = smem + L::wt;
  float* s_mx = smem + L::mx;
  __syncthreads();
  // merge weights of the warps' partials, once per (warp, head)
  if (tid < kWarps * G) {
    const int w = tid / G, h = tid % G;
    float M = -INFINITY;
#pragma unroll
    for (int x = 0; x < kWarps; ++x) M = fmaxf(M, s_m[x * G + h]);
    const float wt = merge_weight(s_m[w * G + h], M);
    s_wt[w * G + h] = wt;
    if (w == 0) s_mx[h] = M;
  }
  __syncthreads();
  cluster_wait();  // every CTA of the cluster has started: CTA 0's shared memory is live
  float* c_m = cluster.map_shared_rank(smem + L::cm, 0);
  float* c_l = cluster.map_shared_rank(smem + L::cl, 0);
  float* c_o = cluster.map_shared_rank(smem + L::co, 0);
  for (int e = tid; e < G * kD; e += T) {
    const int h = e / kD, c = e % kD;
    float O = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) O = fmaf(s_o[(w * G + h) * kD + c], s_wt[w * G + h], O);
    c_o[(crank * G + h) * kD + c] = O;
    if (c == 0) {
      float Ls = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) Ls = fmaf(s_l[w * G + h], s_wt[w * G + h], Ls);
      c_m[crank * G + h] = s_mx[h];
      c_l[crank * G + h] = Ls;
    }
  }
  cluster.sync();  // the pushed partials are visible in CTA 0
  if (crank != 0) return;
  const float* pm = smem + L::cm;
  const float* pl = smem + L::cl;
  const float* po = smem + L::co;
  if (tid < csize * G) {  // merge weights of the CTAs' partials
    const int rk = tid / G, h = tid % G;
    float M = -INFINITY;
    for (int x = 0; x < csize; ++x) M = fmaxf(M, pm[x * G + h]);
    s_wt[rk * G + h] = merge_weight(pm[rk * G + h], M);
  }
  __syncthreads();
  if (tid < G) {
    float Ls = 0.0f;
    for (int rk = 0; rk < csize; ++rk) Ls = fmaf(pl[rk * G + tid], s_wt[rk * G + tid], Ls);
    s_mx[G + tid] = Ls;
  }
  __syncthreads();
  for (int e = tid; e < G * kD; e += T) {
    const int h = e / kD, c = e % kD;
    float O = 0.0f;
    for (int rk = 0; rk < csize; ++rk) O = fmaf(po[(rk * G + h) * kD + c], s_wt[rk * G + h], O);
    const float Ls = s_mx[G + h];
    const float v = Ls > 0.0f ? O / Ls : 0.0f;
    const int64_t qh = int64_t(r) * G + h;
    if (out) out[qh * kD + c] = v;
    if (out_bf16) {
      const __nv_bfloat16 b = __float2bfloat16_rn(v);
      out_bf16[qh * kD + c] = *reinterpret_cast<const uint16_t*>(&b);
    }
  }
}

template <int G, typename KV>
cudaError_t launch_attn_t(int rows, int64_t n, int64_t k, const void* q, int q_dtype, const void* K, const void* V,
                          int64_t stride, int kv_div, const int32_t* idx, float* out, uint16_t* out_bf16,
                          cudaStream_t st) {
  auto kern = attn_cluster_kernel<G, KV>;
  constexpr size_t smem = AttnSmem<G, attn_threads<G>()>::bytes;
  // 16-CTA clusters need an opt-in per kernel; fall back to the portable 8 if it is refused
  static int cluster = 0;
  if (cluster == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    cluster = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess
                  ? kClusterMax
                  : 8;
    cudaGetLastError();
  }
  for (;;) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(cluster), unsigned(rows), 1);
    cfg.blockDim = dim3(attn_threads<G>(), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, n, k, stride, kv_div, q, q_dtype, reinterpret_cast<const KV*>(K),
                                             reinterpret_cast<const KV*>(V), idx, out, out_bf16);
    if (e == cudaSuccess || cluster == 8) return e;
    cudaGetLastError();  // the larger cluster could not be scheduled: use the portable size from now on
    cluster = 8;
  }
}

template <int G>
cudaError_t launch_attn_g(int rows, int64_t n, int64_t k, const void* q, int q_dtype, const void* K, const void* V,
                          int kv_dtype, int64_t stride, const int32_t* idx, float* out, uint16_t* out_bf16,
                          cudaStream_t st, int kv_div = 1) {
  if (kv_dtype == FATHOM_F32)
    return launch_attn_t<G, float>(rows, n, k, q, q_dtype, K, V, stride, kv_div, idx, out, out_bf16, st);
  if (kv_dtype == FATHOM_F16)
    return launch_attn_t<G, __half>(rows, n, k, q, q_dtype, K, V, stride, kv_div, idx, out, out_bf16, st);
  return launch_attn_t<G, __nv_bfloat16>(rows, n, k, q, q_dtype, K, V, stride, kv_div, idx, out, out_bf16, st);
}

}  // namespace

size_t attn_ws_bytes(int, int, int64_t) { return 256; }

cudaError_t launch_attn(int rows, int group, int64_t n, int64_t k, const void* q, int q_dtype, const void* K,
                        const void* V, int kv_dtype, int64_t kv_stride, const int32_t* idx, float* out,
                        uint16_t* out_bf16, void* /*ws*/, cudaStream_t st, bool per_head) {
  if (per_head)  // every query head is a row of its own over its KV row's K/V
    return launch_attn_g<1>(rows * group, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, st,
                            group);
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

static int sparse_attn_impl(int rows, int group, int64_t n, int64_t k, const void* q, int q_dtype, const void* K,
                            const void* V, int kv_dtype, int64_t kv_stride, const int32_t* idx, float* out,
                            uint16_t* out_bf16, void* workspace, size_t ws_bytes, void* stream, bool per_head) {
  clear_error();
  if (rows < 1 || group < 1 || group > 8 || n < 1 || k < 1 || n > 0x7fffffff ||
      int64_t(rows) * (per_head ? group : 1) > 65535)
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
                              (float*)dO, (uint16_t*)dB, const_cast<void*>(dW), as_stream(stream), per_head));
  return FATHOM_OK;
}

int fathom_sparse_attn(int rows, int group, int64_t n, int64_t k, const void* q, int q_dtype, const void* K,
                       const void* V, int kv_dtype, int64_t kv_stride, const int32_t* idx, float* out,
                       uint16_t* out_bf16, void* workspace, size_t ws_bytes, void* stream) {
  return sparse_attn_impl(rows, group, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, workspace,
                          ws_bytes, stream, false);
}

int fathom_sparse_attn_heads(int rows, int group, int64_t n, int64_t k, const void* q, int q_dtype, const void* K,
                             const void* V, int kv_dtype, int64_t kv_stride, const int32_t* idx, float* out,
                             uint16_t* out_bf16, void* workspace, size_t ws_bytes, void* stream) {
  return sparse_attn_impl(rows, group, n, k, q, q_dtype, K, V, kv_dtype, kv_stride, idx, out, out_bf16, workspace,
                          ws_bytes, stream, true);
}

}  // extern "C"
