// fathom_scan: per-query variable-depth scan of the bit-plane index.
//
// Fathom article, "How each query picks its own depth" and "Bit planes: how a
// partial read becomes a valid read": a query reads, for each channel, only
// the first b_c planes (b_c = 0: the channel is skipped and nothing of it is
// read); planes 0..b_c-1 are exactly the b_c-bit quantiser with the channel's
// scale.  The score of key t is
//     s(t) = sum_{c: b_c>=1} qbar_c * (lo + delta*(m*p_c(t) + (m-1)/2)),
// m = 2^(4-b_c), p_c(t) the b_c-bit prefix, (lo, delta) of t's 128-token block.
//
// GPU form.  With the index in HBM the integer work per bit bounds this scan
// (the article's "Where this does not work"; the Rootconf proposal's "What
// made it difficult"), so the kernel is organised around it:
//   * one thread owns 32 consecutive tokens = exactly one 32-bit word of every
//     plane, so a warp reads 128 contiguous bytes per (channel, plane) and
//     never extracts a bit it does not use;
//   * a 4-stage cp.async ring stages each thread's plane words and block
//     (lo, delta) a few channels ahead, hiding memory latency without
//     registers (each thread reads back only what it copied, so no barrier);
//   * per channel, the b_c planes are merged into four "nibble words" (8 tokens
//     x 4 bits) with b_c shifts and b_c-1 bit-select ops each; the prefix of a
//     token becomes the float 1 + u/16 by one shift and one mask-or under the
//     mantissa of 1.0 (exact, mask depends on b_c);
//   * x = fma(16*delta, 1 + u/16, lo + delta*((m-1)/2 - 16)) = lo + delta*(u +
//     (m-1)/2) with a single rounding, then acc += qbar * x; both FMAs run on
//     two tokens at a time (packed f32x2), so each term carries only a few ulps
//     of |qbar_c * x_c| of error.
// Inside the decode step the kernel also builds the 12-bit first-digit
// histogram of its scores for the top-k.
#include "common.cuh"

namespace fathom {
namespace {

constexpr int kScanThreads = 256;  // 8192 tokens per CTA
constexpr int kTokPerThread = 32;
constexpr int kTile = kScanThreads * kTokPerThread;
constexpr int kStages = 4;

template <int SH>
__device__ __forceinline__ uint32_t shift_signed(uint32_t x) {
  // SH > 0: right shift, SH < 0: left shift (compile-time)
  if constexpr (SH > 0) return x >> SH;
  else if constexpr (SH < 0) return x << (-SH);
  else return x;
}

// bit select: bits of a where mask is set, of b elsewhere
__device__ __forceinline__ uint32_t bitsel(uint32_t mask, uint32_t a, uint32_t b) { return (a & mask) | (b & ~mask); }

// o_k for depth DEP: nibble m holds the prefix of token 4m+k in its top DEP bits
// (plane 0 in bit 3); bits below the prefix are left unspecified (masked later).
template <int DEP, int K>
__device__ __forceinline__ uint32_t nibble_word(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
  const uint32_t s0 = shift_signed<K - 3>(w0);
  if constexpr (DEP == 1) return s0;
  const uint32_t s1 = shift_signed<K - 2>(w1);
  if constexpr (DEP == 2) return bitsel(0x88888888u, s0, s1);
  const uint32_t s2 = shift_signed<K - 1>(w2);
  if constexpr (DEP == 3) return bitsel(0x88888888u, s0, bitsel(0x44444444u, s1, s2));
  const uint32_t s3 = shift_signed<K>(w3);
  return bitsel(0x88888888u, s0, bitsel(0x44444444u, s1, bitsel(0x22222222u, s2, s3)));
}

// Mixed-precision FMA (sm_100+): fp16 multiplicands, fp32 addend and result,
// one rounding.  Both fp16 halves of h2 against the same a and c.
__device__ __forceinline__ float2 fma_f16x2_f32(uint16_t a, uint32_t h2, float c) {
  float d0, d1;
  asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "fma.rn.f32.f16 %0, %3, lo, %4;\n\tfma.rn.f32.f16 %1, %3, hi, %4;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "r"(h2), "h"(a), "f"(c));
  return make_float2(d0, d1);
}

// The prefixes of tokens 4M+K (nibble M of o_K) and 4M+16+K (nibble M+4) as two
// fp16 values 16 + u in one register: nibble M -> bits 6..9, nibble M+4 -> bits
// 22..25 (16 apart), under the fp16 exponent of 16 (0x4C00), keeping only the
// prefix bits `mask6` (exact).
template <int M>
__device__ __forceinline__ uint32_t prefix_halves(uint32_t o, uint32_t mask6) {
  return (shift_signed<4 * M - 6>(o) & mask6) | 0x4C004C00u;
}

// x = delta*(16 + u) + lo' = lo + delta*(u + (m-1)/2) in one rounding per token,
// then acc += qbar * x for the two tokens at once (packed f32x2 FMA).
__device__ __forceinline__ void accumulate_halves(float2& acc, uint32_t h2, uint16_t dl16, float lop, float2 q2) {
  const float2 x = fma_f16x2_f32(dl16, h2, lop);
  acc = __ffma2_rn(q2, x, acc);
}

// acc[4m + k] holds tokens (4m + k, 4m + 16 + k).
template <int DEP>
__device__ __forceinline__ void channel_terms(float2 (&acc)[kTokPerThread / 2], uint32_t w0, uint32_t w1, uint32_t w2,
                                              uint32_t w3, uint16_t dl16, float lop, float2 q2) {
  constexpr uint32_t mnib = (0xF0u >> DEP) & 0xFu;  // top DEP bits of a nibble
  constexpr uint32_t mask6 = (mnib << 6) | (mnib << 22);
  const uint32_t o[4] = {nibble_word<DEP, 0>(w0, w1, w2, w3), nibble_word<DEP, 1>(w0, w1, w2, w3),
                         nibble_word<DEP, 2>(w0, w1, w2, w3), nibble_word<DEP, 3>(w0, w1, w2, w3)};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    accumulate_halves(acc[0 + k], prefix_halves<0>(o[k], mask6), dl16, lop, q2);
    accumulate_halves(acc[4 + k], prefix_halves<1>(o[k], mask6), dl16, lop, q2);
    accumulate_halves(acc[8 + k], prefix_halves<2>(o[k], mask6), dl16, lop, q2);
    accumulate_halves(acc[12 + k], prefix_halves<3>(o[k], mask6), dl16, lop, q2);
  }
}

__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <bool kHist>
__global__ void __launch_bounds__(kScanThreads, 4) scan_kernel(const uint32_t* __restrict__ planes,
                                                               const __half2* __restrict__ meta,
                                                               const uint8_t* __restrict__ bits,
                                                               const float* __restrict__ qbar,
                                                               float* __restrict__ scores, uint32_t* __restrict__ hist,
                                                               int64_t n, int64_t nsb, int log2S, int64_t nblk) {
  __shared__ int s_ch[kD];
  __shared__ int s_dep[kD];
  __shared__ float s_q[kD];
  __shared__ int s_wcnt[kD / 32];
  __shared__ uint32_t s_w[kStages][kPlanes][kScanThreads];
  __shared__ __half2 s_m[kStages][kScanThreads];
  __shared__ uint32_t s_hist[kHist ? kHistBins : 1];

  const int r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Active channels of this row, in channel order (warps 0..3, whole warps, cover the 128 channels).
  int dep = 0;
  float qv = 0.0f;
  unsigned ball = 0u;
  if (tid < kD) {
    dep = min(int(bits[int64_t(r) * kD + tid]), kPlanes);
    qv = qbar[int64_t(r) * kD + tid];
    ball = __ballot_sync(0xffffffffu, dep > 0);
    if (lane == 0) s_wcnt[warp] = __popc(ball);
  }
  if constexpr (kHist) {
    for (int i = tid; i < kHistBins; i += kScanThreads) s_hist[i] = 0u;
  }
  __syncthreads();
  int nact = 0;
#pragma unroll
  for (int w = 0; w < kD / 32; ++w) nact += s_wcnt[w];
  if (tid < kD && dep > 0) {
    int off = 0;
    for (int w = 0; w < warp; ++w) off += s_wcnt[w];
    const int pos = off + __popc(ball & ((1u << lane) - 1u));
    s_ch[pos] = tid;
    s_dep[pos] = dep;
    s_q[pos] = qv;
  }
  __syncthreads();

  const int64_t t0 = (int64_t(blockIdx.x) * kScanThreads + tid) * kTokPerThread;
  const bool valid = t0 < n;
  const int64_t S = int64_t(1) << log2S;
  const int64_t run = S >> 5;
  const int64_t tt = valid ? t0 : 0;
  const uint32_t* pb = planes + (int64_t(r) * nsb + (tt >> log2S)) * (kD * kPlanes) * run + ((tt & (S - 1)) >> 5);
  const __half2* mb = meta + int64_t(r) * kD * nblk + (tt >> 7);

  auto issue = [&](int a) {
    if (a < nact && valid) {
      const int st = a % kStages;
      const int c = s_ch[a], d = s_dep[a];
      const uint32_t* p = pb + int64_t(c) * kPlanes * run;
      cp_async4(&s_w[st][0][tid], p);
      if (d > 1) cp_async4(&s_w[st][1][tid], p + run);
      if (d > 2) cp_async4(&s_w[st][2][tid], p + 2 * run);
      if (d > 3) cp_async4(&s_w[st][3][tid], p + 3 * run);
      cp_async4(&s_m[st][tid], mb + int64_t(c) * nblk);
    }
    cp_async_commit();  // one group per channel, possibly empty
  };

  float2 acc[kTokPerThread / 2];  // acc[i] = tokens (i, i + 16) of this thread's 32
#pragma unroll
  for (int i = 0; i < kTokPerThread / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);

#pragma unroll
  for (int a = 0; a < kStages - 1; ++a) issue(a);
  for (int a = 0; a < nact; ++a) {
    issue(a + kStages - 1);
    cp_async_wait<kStages - 1>();  // this thread's copies for channel a have landed
    if (!valid) continue;
    const int st = a % kStages;
    const int d = s_dep[a];
    const float q = s_q[a];
    const __half2 mh = s_m[st][tid];
    const float lo = __low2float(mh), dl = __high2float(mh);
    const uint16_t dl16 = __half_as_ushort(__high2half(mh));
    const float half_m1 = float((1 << (4 - d)) - 1) * 0.5f;  // (m - 1) / 2
    // lo' = lo + delta*((m-1)/2 - 16): exact for fp16 lo, delta unless |lo| > 2^12 delta
    const float lop = fmaf(dl, half_m1 - 16.0f, lo);
    const float2 q2 = make_float2(q, q);
    const uint32_t w0 = s_w[st][0][tid];
    switch (d) {  // uniform across the CTA
      case 1: channel_terms<1>(acc, w0, 0u, 0u, 0u, dl16, lop, q2); break;
      case 2: channel_terms<2>(acc, w0, s_w[st][1][tid], 0u, 0u, dl16, lop, q2); break;
      case 3: channel_terms<3>(acc, w0, s_w[st][1][tid], s_w[st][2][tid], 0u, dl16, lop, q2); break;
      default:
        channel_terms<4>(acc, w0, s_w[st][1][tid], s_w[st][2][tid], s_w[st][3][tid], dl16, lop, q2);
        break;
    }
  }
  cp_async_wait<0>();

  if (valid) {
    float* out = scores + int64_t(r) * n + t0;
    if (t0 + kTokPerThread <= n && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        reinterpret_cast<float4*>(out)[i] =
            make_float4(acc[4 * i].x, acc[4 * i + 1].x, acc[4 * i + 2].x, acc[4 * i + 3].x);
        reinterpret_cast<float4*>(out)[4 + i] =
            make_float4(acc[4 * i].y, acc[4 * i + 1].y, acc[4 * i + 2].y, acc[4 * i + 3].y);
      }
    } else {
#pragma unroll
      for (int i = 0; i < kTokPerThread / 2; ++i) {
        if (t0 + i < n) out[i] = acc[i].x;
        if (t0 + 16 + i < n) out[16 + i] = acc[i].y;
      }
    }
    if constexpr (kHist) {
#pragma unroll
      for (int i = 0; i < kTokPerThread / 2; ++i) {
        if (t0 + i < n) atomicAdd(&s_hist[score_key(acc[i].x) >> (32 - kHistBits)], 1u);
        if (t0 + 16 + i < n) atomicAdd(&s_hist[score_key(acc[i].y) >> (32 - kHistBits)], 1u);
      }
    }
  }
  if constexpr (kHist) {
    __syncthreads();
    uint32_t* gh = hist + int64_t(r) * kHistBins;
    for (int i = tid; i < kHistBins; i += kScanThreads) {
      const uint32_t v = s_hist[i];
      if (v) atomicAdd(gh + i, v);
    }
  }
}

}  // namespace

cudaError_t launch_scan(const IndexGeom& g, const uint32_t* planes, const __half2* meta, const uint8_t* bits,
                        const float* qbar, float* scores, uint32_t* hist, cudaStream_t st) {
  const int64_t tiles = (g.n + kTile - 1) / kTile;
  const dim3 grid{unsigned(tiles), unsigned(g.rows), 1u};
  if (hist)
    scan_kernel<true><<<grid, kScanThreads, 0, st>>>(planes, meta, bits, qbar, scores, hist, g.n, g.nsb, g.log2S,
                                                     g.nblk);
  else
    scan_kernel<false><<<grid, kScanThreads, 0, st>>>(planes, meta, bits, qbar, scores, nullptr, g.n, g.nsb, g.log2S,
                                                      g.nblk);
  return cudaGetLastError();
}

}  // namespace fathom

using namespace fathom;

extern "C" int fathom_scan(const fathom_index_desc* desc, const uint32_t* planes, const uint16_t* meta,
                           const uint8_t* bits, const float* qbar, float* scores, void* stream) {
  clear_error();
  IndexGeom g;
  FATHOM_TRY(index_geom(desc, &g));
  if (g.rows > 65535) return set_error(FATHOM_EINVAL, "rows > 65535");
  const void *dP, *dM, *dB, *dQ, *dS;
  FATHOM_TRY(device_view(planes, "planes", &dP));
  FATHOM_TRY(device_view(meta, "meta", &dM));
  FATHOM_TRY(device_view(bits, "bits", &dB));
  FATHOM_TRY(device_view(qbar, "qbar", &dQ));
  FATHOM_TRY(device_view(scores, "scores", &dS));
  if ((reinterpret_cast<uintptr_t>(dP) & 3) != 0 || (reinterpret_cast<uintptr_t>(dM) & 3) != 0)
    return set_error(FATHOM_EINVAL, "planes and meta must be 4-byte aligned");
  FATHOM_TRY_CUDA(launch_scan(g, (const uint32_t*)dP, (const __half2*)dM, (const uint8_t*)dB, (const float*)dQ,
                              (float*)dS, nullptr, as_stream(stream)));
  return FATHOM_OK;
}
