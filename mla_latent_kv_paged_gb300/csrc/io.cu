// Byte copies for the step's host I/O, done by a kernel: the inputs of a step
// from pinned host buffers into device buffers, and its outputs back. On a
// GB300 the GPU reads and writes pinned host memory over NVLink-C2C; with every
// SM's loads in flight a copy of a megabyte or two finishes well before the
// copy engine's (whose fixed cost dominates at those sizes).
#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n) {
  const size_t stride = (size_t)gridDim.x * kCopyThreads;
  size_t i = (size_t)blockIdx.x * kCopyThreads + threadIdx.x;
  // four loads in flight per thread before their stores
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n; i += stride) dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, cudaStream_t s) {
  const size_t n = bytes / 16;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const size_t want = (n + kCopyThreads - 1) / kCopyThreads;
  const size_t cap = (size_t)sms * 8;  // one wave of 2048 threads per SM
  const unsigned blocks = (unsigned)(want < cap ? want : cap);
  // an ordinary launch: it starts after the kernel before it has finished and
  // the kernel after it starts after it has finished
  copy16_kernel<<<blocks, kCopyThreads, 0, s>>>(reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), n);
  return cudaGetLastError();
}

}  // namespace mla
