// fathom_allocate: per-query reverse water-filling of a bits-per-token budget.
//
// Fathom article, "How each query picks its own depth": a channel's importance
// is the share of score variance it carries; one more bit on a channel removes
// error in proportion to that importance divided by four to the power of the
// bits already spent; the budget goes to the largest such marginal gains (the
// page finds the cut by binary-searching a threshold; selecting the B largest
// gains with a fixed tie order is the same allocation).  Importance of channel c
// is w_c = qbar_c^2 * var_c (Glonce summary: variance-weighted importance).
//
// fathom_allocate_heads takes the same allocation per query head (each head's
// own q_h instead of the summed group query), the alternative reading of GQA.
//
// GPU form: one CTA per row, one thread per candidate (channel c, plane j).
// The threshold tau -- the B-th largest gain -- is found (as on the page, by
// narrowing down a threshold) as a radix select over the bit patterns of the
// non-negative fp32 gains, which order like integers: four passes of 8 bits,
// each a 256-bin histogram of the candidates that match the digits found so far,
// then one warp finding the digit where the count from the top reaches B.
// Gains above tau are taken; gains equal to tau are handed out in (j, c) order
// (j ascending, then c ascending) until exactly B are taken.  The kernel also
// zeroes a span of the caller's workspace (the top-k histogram the scan fills
// next), sparing the step a memset.
#include "common.cuh"

namespace fathom {
namespace {

constexpr int kCand = kD * kPlanes;  // 512 candidates per row

// Row r sums `group` query heads; its variance and budget are those of KV row r / heads
// (heads = 1: one allocation per KV head; group = 1, heads = G: one per query head).
__global__ void __launch_bounds__(kCand) allocate_kernel(int group, int heads, const void* __restrict__ q, int q_dtype,
                                                         const float* __restrict__ var,
                                                         const uint16_t* __restrict__ budgets, int budget,
                                                         uint8_t* __restrict__ bits, float* __restrict__ qbar,
                                                         int32_t* __restrict__ status, uint4* __restrict__ zero,
                                                         int64_t zero16) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < zero16; i += int64_t(gridDim.x) * blockDim.x)
    zero[i] = make_uint4(0u, 0u, 0u, 0u);
  __shared__ float s_gain[kD];
  __shared__ int s_count[kD];
  __shared__ int s_weq[kCand / 32];
  __shared__ int s_bad;
  __shared__ uint32_t s_h[256];
  __shared__ int s_dig[2];  // the digit found, and the matching candidates above it
  const int r = blockIdx.x;
  const int i = threadIdx.x;  // candidate index = j * 128 + c
  const int c = i & (kD - 1), j = i >> 7;
  if (i == 0) s_bad = 0;
  if (i < kD) s_count[i] = 0;
  __syncthreads();
  float w = 0.0f;
  if (j == 0) {
    const int64_t q0 = int64_t(r) * group * kD + c;
    float s = load_as_float(q, q0, q_dtype);
    for (int h = 1; h < group; ++h) s = __fadd_rn(s, load_as_float(q, q0 + int64_t(h) * kD, q_dtype));
    const float v = var[int64_t(r / heads) * kD + c];
    qbar[int64_t(r) * kD + c] = s;
    // + 0 turns a -0 product (var = -0) into +0: equal gains need equal bit patterns
    w = __fadd_rn(__fmul_rn(__fmul_rn(s, s), v), 0.0f);
    // a variance is never negative; an importance that overflows has no order
    if (!isfinite(s) || !isfinite(v) || v < 0.0f || !isfinite(w)) s_bad = 1;
    s_gain[c] = w;
  }
  __syncthreads();
  if (s_bad) {
    if (i < kD) bits[int64_t(r) * kD + i] = 0;
    if (i == 0 && status) atomicOr(status, FATHOM_STATUS_NONFINITE);
    return;
  }
  if (j > 0) {
    w = s_gain[c];
    for (int jj = 0; jj < j; ++jj) w = __fmul_rn(w, 0.25f);
  }
  const uint32_t gb = __float_as_uint(w);  // w >= +0: bit patterns order like the values
  int B = budgets ? int(budgets[r / heads]) : budget;
  if (B > kCand) {
    if (i == 0 && status) atomicOr(status, FATHOM_STATUS_BUDGET_CLAMPED);
    B = kCand;
  }
  bool take = false;
  if (B > 0) {
    // radix select of the B-th largest gain, 8 bits a pass from the top
    uint32_t prefix = 0u, pmask = 0u;
    int need = B;  // gains still to reach among those matching prefix under pmask
#pragma unroll 1
    for (int sh = 24; sh >= 0; sh -= 8) {
      if (i < 256) s_h[i] = 0u;
      __syncthreads();
      if ((gb & pmask) == prefix) atomicAdd(&s_h[(gb >> sh) & 255u], 1u);
      __syncthreads();
      if (i < 32) {  // lane l holds bins 255 - 8l .. 248 - 8l (descending)
        int bins[8], sum = 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          bins[b] = int(s_h[255 - 8 * i - b]);
          sum += bins[b];
        }
        int cum = sum;  // inclusive scan over the lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, cum, o);
          if (i >= o) cum += y;
        }
        int before = cum - sum;
        if (before < need && cum >= need) {
          int b = 0;
          for (; b < 7; ++b) {
            if (before + bins[b] >= need) break;
            before += bins[b];
          }
          s_dig[0] = 255 - 8 * i - b;
          s_dig[1] = before;
        }
      }
      __syncthreads();
      need -= s_dig[1];
      prefix |= uint32_t(s_dig[0]) << sh;
      pmask |= 255u << sh;
    }
    const uint32_t lo = prefix;  // tau: B - need gains lie above it
    const int above = B - need;
    // rank of this candidate among those equal to tau, in (j, c) order = thread order
    const unsigned eqb = __ballot_sync(0xffffffffu, gb == lo);
    if ((i & 31) == 0) s_weq[i >> 5] = __popc(eqb);
    __syncthreads();
    int eq_before = __popc(eqb & ((1u << (i & 31)) - 1u));
    for (int wp = 0; wp < (i >> 5); ++wp) eq_before += s_weq[wp];
    take = gb > lo || (gb == lo && eq_before < B - above);
  }
  if (take) atomicAdd(&s_count[c], 1);
  __syncthreads();
  if (i < kD) bits[int64_t(r) * kD + i] = uint8_t(s_count[i]);
}

// SparQ-style comparator: full depth on the r channels of largest |qbar| (ties
// to the lower channel), nothing elsewhere.  One CTA per row, one thread per channel.
__global__ void __launch_bounds__(kD) allocate_sparq_kernel(int group, const void* __restrict__ q, int q_dtype,
                                                            int r_channels, uint8_t* __restrict__ bits,
                                                            float* __restrict__ qbar, int32_t* __restrict__ status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  __shared__ float s_a[kD];
  const int r = blockIdx.x, c = threadIdx.x;
  const int64_t q0 = int64_t(r) * group * kD + c;
  float s = load_as_float(q, q0, q_dtype);
  for (int h = 1; h < group; ++h) s = __fadd_rn(s, load_as_float(q, q0 + int64_t(h) * kD, q_dtype));
  qbar[int64_t(r) * kD + c] = s;
  const float a = fabsf(s);
  s_a[c] = a;
  const int bad = __syncthreads_or(!isfinite(s));
  if (bad) {
    bits[int64_t(r) * kD + c] = 0;
    if (c == 0 && status) atomicOr(status, FATHOM_STATUS_NONFINITE);
    return;
  }
  int rank = 0;
  for (int o = 0; o < kD; ++o) rank += (s_a[o] > a) || (s_a[o] == a && o < c);
  bits[int64_t(r) * kD + c] = rank < r_channels ? uint8_t(kPlanes) : uint8_t(0);
}

__global__ void __launch_bounds__(kD) qbar_kernel(int group, const void* __restrict__ q, int q_dtype,
                                                  float* __restrict__ qbar) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_trigger();
  const int r = blockIdx.x, c = threadIdx.x;
  const int64_t q0 = int64_t(r) * group * kD + c;
  float s = load_as_float(q, q0, q_dtype);
  for (int h = 1; h < group; ++h) s = __fadd_rn(s, load_as_float(q, q0 + int64_t(h) * kD, q_dtype));
  qbar[int64_t(r) * kD + c] = s;
}

}  // namespace

cudaError_t launch_allocate(int rows, int group, const void* q, int q_dtype, const float* var, const uint16_t* budgets,
                            int budget, uint8_t* bits, float* qbar, int32_t* status, cudaStream_t st, void* zero,
                            size_t zero_bytes) {
  if ((reinterpret_cast<uintptr_t>(zero) | zero_bytes) & 15) return cudaErrorInvalidValue;
  return pdl_launch(allocate_kernel, dim3(rows), dim3(kCand), 0, st, group, 1, q, q_dtype, var, budgets, budget, bits,
                    qbar, status, static_cast<uint4*>(zero), int64_t(zero_bytes / 16));
}

cudaError_t launch_allocate_heads(int rows, int group, const void* q, int q_dtype, const float* var,
                                  const uint16_t* budgets, int budget, uint8_t* bits, float* qh, int32_t* status,
                                  cudaStream_t st) {
  return pdl_launch(allocate_kernel, dim3(rows * group), dim3(kCand), 0, st, 1, group, q, q_dtype, var, budgets,
                    budget, bits, qh, status, static_cast<uint4*>(nullptr), int64_t(0));
}

cudaError_t launch_allocate_sparq(int rows, int group, const void* q, int q_dtype, int r_channels, uint8_t* bits,
                                  float* qbar, int32_t* status, cudaStream_t st) {
  return pdl_launch(allocate_sparq_kernel, dim3(rows), dim3(kD), 0, st, group, q, q_dtype, r_channels, bits, qbar,
                    status);
}

cudaError_t launch_qbar(int rows, int group, const void* q, int q_dtype, float* qbar, cudaStream_t st) {
  return pdl_launch(qbar_kernel, dim3(rows), dim3(kD), 0, st, group, q, q_dtype, qbar);
}

}  // namespace fathom

using namespace fathom;

extern "C" int fathom_allocate(int rows, int group, const void* q, int q_dtype, const float* var,
                               const uint16_t* budgets, int budget, uint8_t* bits, float* qbar, int32_t* status,
                               void* stream) {
  clear_error();
  if (rows < 1 || group < 1 || group > 64) return set_error(FATHOM_EINVAL, "rows >= 1 and 1 <= group <= 64 required");
  if (!valid_dtype(q_dtype)) return set_error(FATHOM_EINVAL, "q_dtype %d invalid", q_dtype);
  if (!budgets && (budget < 0 || budget > kD * kPlanes))
    return set_error(FATHOM_EINVAL, "budget %d outside [0, 512]", budget);
  const void *dq, *dv, *db, *dbits, *dqb, *dst;
  FATHOM_TRY(device_view(q, "q", &dq));
  FATHOM_TRY(device_view(var, "var", &dv));
  FATHOM_TRY(device_view(budgets, "budgets", &db, true));
  FATHOM_TRY(device_view(bits, "bits", &dbits));
  FATHOM_TRY(device_view(qbar, "qbar", &dqb));
  FATHOM_TRY(device_view(status, "status", &dst, true));
  FATHOM_TRY_CUDA(launch_allocate(rows, group, dq, q_dtype, (const float*)dv, (const uint16_t*)db, budget,
                                  (uint8_t*)dbits, (float*)dqb, (int32_t*)dst, as_stream(stream)));
  return FATHOM_OK;
}

extern "C" int fathom_allocate_heads(int rows, int group, const void* q, int q_dtype, const float* var,
                                     const uint16_t* budgets, int budget, uint8_t* bits, float* qh, int32_t* status,
                                     void* stream) {
  clear_error();
  if (rows < 1 || group < 1 || group > 64 || int64_t(rows) * group > 0x7fffffff)
    return set_error(FATHOM_EINVAL, "rows >= 1 and 1 <= group <= 64 required");
  if (!valid_dtype(q_dtype)) return set_error(FATHOM_EINVAL, "q_dtype %d invalid", q_dtype);
  if (!budgets && (budget < 0 || budget > kD * kPlanes))
    return set_error(FATHOM_EINVAL, "budget %d outside [0, 512]", budget);
  const void *dq, *dv, *db, *dbits, *dqh, *dst;
  FATHOM_TRY(device_view(q, "q", &dq));
  FATHOM_TRY(device_view(var, "var", &dv));
  FATHOM_TRY(device_view(budgets, "budgets", &db, true));
  FATHOM_TRY(device_view(bits, "bits", &dbits));
  FATHOM_TRY(device_view(qh, "qh", &dqh));
  FATHOM_TRY(device_view(status, "status", &dst, true));
  FATHOM_TRY_CUDA(launch_allocate_heads(rows, group, dq, q_dtype, (const float*)dv, (const uint16_t*)db, budget,
                                        (uint8_t*)dbits, (float*)dqh, (int32_t*)dst, as_stream(stream)));
  return FATHOM_OK;
}

extern "C" int fathom_allocate_sparq(int rows, int group, const void* q, int q_dtype, int r_channels, uint8_t* bits,
                                     float* qbar, int32_t* status, void* stream) {
  clear_error();
  if (rows < 1 || group < 1 || group > 64) return set_error(FATHOM_EINVAL, "rows >= 1 and 1 <= group <= 64 required");
  if (!valid_dtype(q_dtype)) return set_error(FATHOM_EINVAL, "q_dtype %d invalid", q_dtype);
  if (r_channels < 0 || r_channels > kD) return set_error(FATHOM_EINVAL, "r_channels %d outside [0, 128]", r_channels);
  const void *dq, *dbits, *dqb, *dst;
  FATHOM_TRY(device_view(q, "q", &dq));
  FATHOM_TRY(device_view(bits, "bits", &dbits));
  FATHOM_TRY(device_view(qbar, "qbar", &dqb));
  FATHOM_TRY(device_view(status, "status", &dst, true));
  FATHOM_TRY_CUDA(launch_allocate_sparq(rows, group, dq, q_dtype, r_channels, (uint8_t*)dbits, (float*)dqb,
                                        (int32_t*)dst, as_stream(stream)));
  return FATHOM_OK;
}
