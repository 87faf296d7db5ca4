// fathom_probe_stream_read: streaming-read bandwidth of HBM or of the host link
// (zero-copy loads of pinned, mapped host memory), used as the measured peak
// beside the scan's achieved bandwidth.
// fathom_probe_int_ops: the integer ALU rate (shifts and bit selects, the work
// of bit extraction), for the machine balance of integer operations per byte.
#include "../../include/fathom_probe.h"
#include "common.cuh"

namespace fathom {
namespace {

__global__ void stream_read_kernel(const uint4* __restrict__ p, size_t n16, uint32_t* __restrict__ sink) {
  uint32_t acc = 0u;
  const size_t stride = size_t(gridDim.x) * blockDim.x;
#pragma unroll 4
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 v = __ldg(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  acc = __reduce_xor_sync(0xffffffffu, acc);
  if ((threadIdx.x & 31) == 0 && acc != 0u) atomicXor(sink, acc);
}

// 8 independent chains per thread; each step of a chain is two right shifts and
// one three-input XOR: 3 ALU-pipe instructions (right shifts cannot move to the
// FMA pipe as multiplies).
__global__ void int_ops_kernel(int iters, uint32_t seed, uint32_t* __restrict__ sink) {
  uint32_t x[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = seed + (blockIdx.x * blockDim.x + threadIdx.x) * 8u + uint32_t(j);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = (x[j] >> 3) ^ (x[j] >> 11) ^ (0x9E3779B9u + uint32_t(j));
  }
  uint32_t acc = 0u;
#pragma unroll
  for (int j = 0; j < 8; ++j) acc ^= x[j];
  if (acc == 0x5EED1234u) atomicAdd(sink, 1u);  // keeps the chains live
}

}  // namespace
}  // namespace fathom

using namespace fathom;

extern "C" int fathom_probe_stream_read(const void* buf, size_t bytes, int blocks_per_sm, int threads,
                                        uint32_t* sink, void* stream) {
  clear_error();
  if (bytes == 0 || (bytes & 15) || blocks_per_sm < 1 || blocks_per_sm > 64 || threads < 32 || threads > 1024 ||
      (threads & 31))
    return set_error(FATHOM_EINVAL, "bytes must be a positive multiple of 16; 1 <= blocks_per_sm <= 64; "
                                    "threads a multiple of 32 up to 1024");
  const void *dB, *dS;
  FATHOM_TRY(device_view(buf, "buf", &dB));
  FATHOM_TRY(device_view(sink, "sink", &dS));
  if (reinterpret_cast<uintptr_t>(dB) & 15) return set_error(FATHOM_EINVAL, "buf must be 16-byte aligned");
  stream_read_kernel<<<blocks_per_sm * num_sms(), threads, 0, as_stream(stream)>>>(
      reinterpret_cast<const uint4*>(dB), bytes / 16, (uint32_t*)dS);
  FATHOM_TRY_CUDA(cudaGetLastError());
  return FATHOM_OK;
}

extern "C" int fathom_probe_int_ops(int iters, int blocks_per_sm, int threads, uint32_t* sink, void* stream) {
  clear_error();
  if (iters < 1 || blocks_per_sm < 1 || blocks_per_sm > 64 || threads < 32 || threads > 1024 || (threads & 31))
    return set_error(FATHOM_EINVAL, "iters >= 1; 1 <= blocks_per_sm <= 64; threads a multiple of 32 up to 1024");
  const void* dS;
  FATHOM_TRY(device_view(sink, "sink", &dS));
  int_ops_kernel<<<blocks_per_sm * num_sms(), threads, 0, as_stream(stream)>>>(iters, 12345u, (uint32_t*)dS);
  FATHOM_TRY_CUDA(cudaGetLastError());
  return FATHOM_OK;
}

extern "C" int fathom_probe_num_sms(void) { return num_sms(); }
