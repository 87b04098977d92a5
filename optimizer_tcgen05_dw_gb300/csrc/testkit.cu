// Test kit (separate library, loaded only by the GPU tests): evaluates the
// device Philox4x32-10 of optim.cuh, and cuRAND's Philox4_32_10 generator, on
// caller-given (counter, key) pairs so the two can be compared with each other
// and with the CPU oracle; and holds SMs for a bounded time, so that a test
// can launch a kernel that does not find the whole device free.
#include <curand_kernel.h>

#include "optim.cuh"

namespace {

// in: n x 6 words (c0, c1, c2, c3, k0, k1); out: n x 4 words.
__global__ void philox_kernel(const uint32_t* in, uint32_t* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t* q = in + 6 * i;
  const uint4 r = forge::dev::philox4x32_10(make_uint4(q[0], q[1], q[2], q[3]), q[4], q[5]);
  out[4 * i] = r.x;
  out[4 * i + 1] = r.y;
  out[4 * i + 2] = r.z;
  out[4 * i + 3] = r.w;
}

// cuRAND: key = seed, counter words (2, 3) = subsequence, words (0, 1) =
// offset / 4; the first curand4() returns the block at that counter.
__global__ void curand_kernel_eval(const uint32_t* in, uint32_t* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t* q = in + 6 * i;
  const unsigned long long seed = (static_cast<unsigned long long>(q[5]) << 32) | q[4];
  const unsigned long long subseq = (static_cast<unsigned long long>(q[3]) << 32) | q[2];
  const unsigned long long ctr01 = (static_cast<unsigned long long>(q[1]) << 32) | q[0];
  curandStatePhilox4_32_10_t st;
  curand_init(seed, subseq, 0ull, &st);
  skipahead(ctr01 * 4ull, &st);
  const uint4 r = curand4(&st);
  out[4 * i] = r.x;
  out[4 * i + 1] = r.y;
  out[4 * i + 2] = r.z;
  out[4 * i + 3] = r.w;
}

// Each block takes its dynamic shared memory (sized by the caller so that no
// large block fits beside it on the SM) and waits on the global timer for `ns`
// nanoseconds, then exits: a bounded wait on nothing but the clock.
__global__ void hold_kernel(uint64_t ns) {
  extern __shared__ uint8_t held[];
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  do {
    __nanosleep(1000);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < ns);
  if (threadIdx.x == 0 && ns == 0) held[0] = 1;  // the buffer stays part of the kernel
}

}  // namespace

extern "C" {

// Holds `blocks` SMs (one block each, `smem` bytes of shared memory) for `ns`
// nanoseconds (at most 2 s) on `stream`.
__attribute__((visibility("default"))) int forge_testkit_hold_sms(int blocks, unsigned long long ns, int smem,
                                                                   void* stream) {
  if (blocks <= 0 || ns > 2000000000ull || smem < 0) return static_cast<int>(cudaErrorInvalidValue);
  cudaError_t e = cudaFuncSetAttribute(hold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return static_cast<int>(e);
  hold_kernel<<<blocks, 32, static_cast<size_t>(smem), static_cast<cudaStream_t>(stream)>>>(ns);
  return static_cast<int>(cudaGetLastError());
}

__attribute__((visibility("default"))) int forge_testkit_philox(const uint32_t* in, uint32_t* out,
                                                                 int n, void* stream) {
  philox_kernel<<<(n + 127) / 128, 128, 0, static_cast<cudaStream_t>(stream)>>>(in, out, n);
  return static_cast<int>(cudaGetLastError());
}

__attribute__((visibility("default"))) int forge_testkit_curand_philox(const uint32_t* in,
                                                                       uint32_t* out, int n,
                                                                       void* stream) {
  curand_kernel_eval<<<(n + 127) / 128, 128, 0, static_cast<cudaStream_t>(stream)>>>(in, out, n);
  return static_cast<int>(cudaGetLastError());
}

}  // extern "C"
