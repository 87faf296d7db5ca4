// Pinned host memory backed by transparent huge pages, for host-resident
// index and K/V stores (fathom_host_alloc / fathom_host_free).
#include <string.h>
#include <sys/mman.h>

#include "common.cuh"

using namespace fathom;

extern "C" {

int fathom_host_alloc(size_t bytes, void** ptr) {
  clear_error();
  if (!ptr || bytes == 0) return set_error(FATHOM_EINVAL, "bytes must be > 0 and ptr non-NULL");
  *ptr = nullptr;
  void* p = mmap(nullptr, bytes, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
  if (p == MAP_FAILED) return set_error(FATHOM_ENOMEM, "mmap of %zu bytes failed", bytes);
#ifdef MADV_HUGEPAGE
  madvise(p, bytes, MADV_HUGEPAGE);  // advisory: without THP the memory is still usable
#endif
  memset(p, 0, bytes);  // populate before registration
  cudaError_t e = cudaHostRegister(p, bytes, cudaHostRegisterMapped | cudaHostRegisterPortable);
  if (e != cudaSuccess) {
    cudaGetLastError();
    munmap(p, bytes);
    return set_error(FATHOM_ENOMEM, "cudaHostRegister of %zu bytes failed: %s", bytes, cudaGetErrorString(e));
  }
  *ptr = p;
  return FATHOM_OK;
}

int fathom_host_free(void* ptr, size_t bytes) {
  clear_error();
  if (!ptr || bytes == 0) return set_error(FATHOM_EINVAL, "ptr and bytes required");
  cudaError_t e = cudaHostUnregister(ptr);
  const int rc = munmap(ptr, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return set_error(FATHOM_ECUDA, "cudaHostUnregister: %s", cudaGetErrorString(e));
  }
  if (rc != 0) return set_error(FATHOM_EINVAL, "munmap failed");
  return FATHOM_OK;
}

}  // extern "C"
