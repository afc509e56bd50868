// Does a device-to-device copy progress while a kernel holds every SM?
//
// A "hog" kernel takes all SMs (one 192-thread block per SM, 225 KB of
// shared memory and about 245 registers per thread, i.e. most of each SM's
// register file) and spins -- for one second at most -- until a flag turns
// non-zero.  On a second stream the probe enqueues a copy and then writes
// the flag with a stream memory operation.  If the copy runs on a copy
// engine the flag arrives within microseconds; if the copy needs an SM it
// cannot start until the hog gives up, and the hog reports the timeout.
//
// Prints one line per copy form: "<form> <microseconds or BLOCKED>".
#include <cstdint>
#include <cstdio>
#include <cuda.h>
#include <cuda_runtime.h>

constexpr int kRegs = 236;               // live floats per thread (about 245 registers)
constexpr size_t kSmem = 225 * 1024;     // dynamic shared memory per block
constexpr uint64_t kLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__global__ void __launch_bounds__(192, 1) hog(const volatile uint32_t* flag, unsigned long long* waited) {
  extern __shared__ float scratch[];
  float live[kRegs];
#pragma unroll
  for (int i = 0; i < kRegs; ++i) live[i] = threadIdx.x * 1e-3f + i;
  const uint64_t t0 = now_ns();
  unsigned long long result = ~0ull;
  for (;;) {
#pragma unroll
    for (int i = 0; i < kRegs; ++i) live[i] = fmaf(live[i], 0.999f, 1e-3f);
    if (*flag != 0) { result = now_ns() - t0; break; }
    if (now_ns() - t0 > kLimitNs) break;
  }
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < kRegs; ++i) sum += live[i];
  scratch[threadIdx.x] = sum;  // keeps the registers live
  __syncthreads();
  if (threadIdx.x == 0) atomicMax(waited, scratch[0] == -1.f ? 0ull : result);
}

typedef CUresult (*WriteValue32)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

int main() {
  WriteValue32 write32 = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", (void**)&write32, 12000, cudaEnableDefault, &q) !=
          cudaSuccess || !write32) {
    printf("no cuStreamWriteValue32\n");
    return 2;
  }
  if (cudaFuncSetAttribute(hog, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) != cudaSuccess) return 2;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const size_t bytes = 4u << 20, row = 4096;
  uint32_t* flag;
  unsigned long long* waited;
  void *src, *dst;
  if (cudaMalloc(&flag, 4) || cudaMalloc(&waited, 8) || cudaMalloc(&src, bytes) || cudaMalloc(&dst, bytes)) return 2;
  cudaStream_t s_hog, s_copy;
  cudaStreamCreateWithFlags(&s_hog, cudaStreamNonBlocking);
  cudaStreamCreateWithFlags(&s_copy, cudaStreamNonBlocking);
  const char* forms[] = {"flag_only", "memcpy_2d", "memcpy_1d"};
  for (int f = 0; f < 3; ++f) {
    cudaMemset(flag, 0, 4);
    cudaMemset(waited, 0, 8);
    cudaDeviceSynchronize();
    hog<<<sms, 192, kSmem, s_hog>>>(flag, waited);
    if (f == 1) cudaMemcpy2DAsync(dst, row, src, row, row, bytes / row, cudaMemcpyDeviceToDevice, s_copy);
    if (f == 2) cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, s_copy);
    write32(s_copy, (CUdeviceptr)flag, 1, 0);
    if (cudaDeviceSynchronize() != cudaSuccess) {
      printf("%s ERROR\n", forms[f]);
      return 1;
    }
    unsigned long long w = 0;
    cudaMemcpy(&w, waited, 8, cudaMemcpyDeviceToHost);
    if (w == ~0ull)
      printf("%s BLOCKED\n", forms[f]);
    else
      printf("%s %llu\n", forms[f], w / 1000);
  }
  return 0;
}
