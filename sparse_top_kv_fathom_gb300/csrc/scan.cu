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
// GPU form (integer work per bit is what bounds this scan when the index sits
// in HBM, per the article's "Where this does not work" and the Rootconf
// proposal): one thread owns 32 consecutive tokens, i.e. exactly one 32-bit
// word of every plane.  For each active channel it loads b_c words (coalesced:
// a warp reads 128 contiguous bytes per plane), merges them into four
// "nibble words" of 8 tokens each with shifts and masks (~1/4 integer op per
// plane bit), then turns each 4-bit prefix into a float by OR-ing it under the
// mantissa of 1.0 (1 + u/16, exact) and accumulates with one FMA per token and
// channel.  The constant part of every term (lo, the bucket centre and the
// -16*delta offset of the 1 + u/16 form) is folded into one per-thread value.
#include "common.cuh"

namespace fathom {
namespace {

constexpr int kScanThreads = 128;                  // one warp group: 4096 tokens per CTA
constexpr int kTokPerThread = 32;
constexpr int kTile = kScanThreads * kTokPerThread;

template <int SH>
__device__ __forceinline__ uint32_t shift_signed(uint32_t x) {
  // SH > 0: right shift, SH < 0: left shift (compile-time)
  if constexpr (SH > 0) return x >> SH;
  else if constexpr (SH < 0) return x << (-SH);
  else return x;
}

// o_k: nibble m holds the 4-bit prefix of token 4m+k (plane 0 in bit 3).
template <int K>
__device__ __forceinline__ uint32_t nibble_word(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
  return (shift_signed<K - 3>(w0) & 0x88888888u) | (shift_signed<K - 2>(w1) & 0x44444444u) |
         (shift_signed<K - 1>(w2) & 0x22222222u) | (shift_signed<K>(w3) & 0x11111111u);
}

// float 1 + u/16 for the nibble M of o (u in 0..15), exact.
template <int M>
__device__ __forceinline__ float nibble_float(uint32_t o) {
  return __uint_as_float((shift_signed<4 * M - 19>(o) & 0x00780000u) | 0x3F800000u);
}

template <int M>
__device__ __forceinline__ float2 nibble_pair(uint32_t oa, uint32_t ob) {
  return make_float2(nibble_float<M>(oa), nibble_float<M>(ob));
}

// Tokens 4m+k0 and 4m+k0+1 (nibble m of oa and ob): x = lo' + 16*delta*(1 + u/16)
// = lo + delta*(u + (m_c - 1)/2) with one rounding, then acc += qbar * x; two
// tokens per packed f32x2 instruction.
template <int M>
__device__ __forceinline__ void accumulate_pair(float2& acc, uint32_t oa, uint32_t ob, float2 d16, float2 lo2,
                                                float2 q2) {
  const float2 x = __ffma2_rn(d16, nibble_pair<M>(oa, ob), lo2);
  acc = __ffma2_rn(q2, x, acc);
}

template <bool kHist>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(const uint32_t* __restrict__ planes,
                                                            const __half2* __restrict__ meta,
                                                            const uint8_t* __restrict__ bits,
                                                            const float* __restrict__ qbar, float* __restrict__ scores,
                                                            uint32_t* __restrict__ hist, int64_t n, int64_t nsb,
                                                            int log2S, int64_t nblk) {
  __shared__ int s_ch[kD];
  __shared__ int s_dep[kD];
  __shared__ float s_q[kD];
  __shared__ int s_wcnt[kScanThreads / 32];
  __shared__ float s_tr[kScanThreads / 32][32][33];
  __shared__ uint32_t s_hist[kHist ? kHistBins : 1];

  const int r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // Active channels of this row, in channel order.
  const int dep = min(int(bits[int64_t(r) * kD + tid]), kPlanes);
  const float qv = qbar[int64_t(r) * kD + tid];
  const unsigned ball = __ballot_sync(0xffffffffu, dep > 0);
  if (lane == 0) s_wcnt[warp] = __popc(ball);
  if constexpr (kHist) {
    for (int i = tid; i < kHistBins; i += kScanThreads) s_hist[i] = 0u;
  }
  __syncthreads();
  int off = 0, nact = 0;
#pragma unroll
  for (int w = 0; w < kScanThreads / 32; ++w) {
    off += (w < warp) ? s_wcnt[w] : 0;
    nact += s_wcnt[w];
  }
  if (dep > 0) {
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

  float2 acc[kTokPerThread / 2];  // acc[i] = tokens (2i, 2i+1)
#pragma unroll
  for (int i = 0; i < kTokPerThread / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);

  for (int a = 0; a < nact; ++a) {
    const int c = s_ch[a];
    const int d = s_dep[a];
    const float q = s_q[a];
    uint32_t w0 = 0u, w1 = 0u, w2 = 0u, w3 = 0u;
    float lo = 0.0f, dl = 0.0f;
    if (valid) {
      const uint32_t* p = pb + int64_t(c) * kPlanes * run;
      w0 = __ldg(p);
      if (d > 1) w1 = __ldg(p + run);
      if (d > 2) w2 = __ldg(p + 2 * run);
      if (d > 3) w3 = __ldg(p + 3 * run);
      const float2 m = __half22float2(__ldg(mb + int64_t(c) * nblk));
      lo = m.x;
      dl = m.y;
    }
    const float half_m1 = float((1 << (4 - d)) - 1) * 0.5f;  // (m - 1) / 2
    // lo' = lo + delta*((m-1)/2 - 16): exact for fp16 lo, delta unless |lo| > 2^12 delta
    const float lop = fmaf(dl, half_m1 - 16.0f, lo);
    const float2 lo2 = make_float2(lop, lop);
    const float2 d16 = make_float2(16.0f * dl, 16.0f * dl);
    const float2 q2 = make_float2(q, q);
    const uint32_t o0 = nibble_word<0>(w0, w1, w2, w3), o1 = nibble_word<1>(w0, w1, w2, w3);
    const uint32_t o2 = nibble_word<2>(w0, w1, w2, w3), o3 = nibble_word<3>(w0, w1, w2, w3);
    accumulate_pair<0>(acc[0], o0, o1, d16, lo2, q2);
    accumulate_pair<0>(acc[1], o2, o3, d16, lo2, q2);
    accumulate_pair<1>(acc[2], o0, o1, d16, lo2, q2);
    accumulate_pair<1>(acc[3], o2, o3, d16, lo2, q2);
    accumulate_pair<2>(acc[4], o0, o1, d16, lo2, q2);
    accumulate_pair<2>(acc[5], o2, o3, d16, lo2, q2);
    accumulate_pair<3>(acc[6], o0, o1, d16, lo2, q2);
    accumulate_pair<3>(acc[7], o2, o3, d16, lo2, q2);
    accumulate_pair<4>(acc[8], o0, o1, d16, lo2, q2);
    accumulate_pair<4>(acc[9], o2, o3, d16, lo2, q2);
    accumulate_pair<5>(acc[10], o0, o1, d16, lo2, q2);
    accumulate_pair<5>(acc[11], o2, o3, d16, lo2, q2);
    accumulate_pair<6>(acc[12], o0, o1, d16, lo2, q2);
    accumulate_pair<6>(acc[13], o2, o3, d16, lo2, q2);
    accumulate_pair<7>(acc[14], o0, o1, d16, lo2, q2);
    accumulate_pair<7>(acc[15], o2, o3, d16, lo2, q2);
  }

  // Transpose through shared memory so that the stores are coalesced.
#pragma unroll
  for (int i = 0; i < kTokPerThread / 2; ++i) {
    s_tr[warp][lane][2 * i] = acc[i].x;
    s_tr[warp][lane][2 * i + 1] = acc[i].y;
  }
  __syncwarp();
  const int64_t tw = (int64_t(blockIdx.x) * kScanThreads + warp * 32) * kTokPerThread;  // warp's first token
  float* out = scores + int64_t(r) * n;
#pragma unroll 4
  for (int i = 0; i < 32; ++i) {
    const int64_t t = tw + int64_t(i) * 32 + lane;
    const float s = s_tr[warp][i][lane];
    if (t < n) {
      out[t] = s;
      if constexpr (kHist) atomicAdd(&s_hist[score_key(s) >> (32 - kHistBits)], 1u);
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
  dim3 grid(unsigned(tiles), unsigned(g.rows));
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
