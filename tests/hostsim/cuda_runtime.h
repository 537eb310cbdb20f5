/* Host-only stand-in for the CUDA runtime, for the host-runtime tests
 * (tests/test_host_runtime.py): it lets the library's host code (api.cu) be
 * compiled with a plain C++ compiler and run without a GPU, so that its
 * bookkeeping -- page allocation, prefix sharing, argument and state checks,
 * error codes -- can be tested on the CPU.  "Device" memory is host memory,
 * copies are memcpy, streams and events do nothing, and every kernel
 * launcher is a stub (tests/hostsim/stubs.cpp).  Never part of the library
 * build. */
#pragma once

#include <cstddef>
#include <cstdlib>
#include <cstring>

#define __host__
#define __device__
#define __global__
#define __align__(n) __attribute__((aligned(n)))

enum cudaError_t { cudaSuccess = 0, cudaErrorInvalidValue = 1, cudaErrorMemoryAllocation = 2 };
typedef cudaError_t cudaError;
enum cudaMemcpyKind {
  cudaMemcpyHostToHost = 0,
  cudaMemcpyHostToDevice = 1,
  cudaMemcpyDeviceToHost = 2,
  cudaMemcpyDeviceToDevice = 3,
  cudaMemcpyDefault = 4
};
enum cudaDeviceAttr { cudaDevAttrMultiProcessorCount = 16 };
typedef struct CUstream_st* cudaStream_t;
typedef struct CUevent_st* cudaEvent_t;

struct dim3 {
  unsigned x, y, z;
  dim3(unsigned a = 1, unsigned b = 1, unsigned c = 1) : x(a), y(b), z(c) {}
};

enum cudaLaunchAttributeID { cudaLaunchAttributeProgrammaticStreamSerialization = 5 };
struct cudaLaunchAttributeValue {
  int programmaticStreamSerializationAllowed;
};
struct cudaLaunchAttribute {
  cudaLaunchAttributeID id;
  cudaLaunchAttributeValue val;
};
struct cudaLaunchConfig_t {
  dim3 gridDim, blockDim;
  size_t dynamicSmemBytes;
  cudaStream_t stream;
  cudaLaunchAttribute* attrs;
  unsigned numAttrs;
};
template <typename... K, typename... A>
inline cudaError_t cudaLaunchKernelEx(const cudaLaunchConfig_t*, void (*)(K...), A...) {
  return cudaSuccess;
}

inline const char* cudaGetErrorString(cudaError_t e) { return e == cudaSuccess ? "no error" : "host stand-in error"; }

inline cudaError_t cudaMalloc(void** p, size_t n) {
  *p = std::aligned_alloc(256, (n + 255) / 256 * 256);
  return *p ? cudaSuccess : cudaErrorMemoryAllocation;
}
template <typename T>
inline cudaError_t cudaMalloc(T** p, size_t n) {
  return cudaMalloc(reinterpret_cast<void**>(p), n);
}
inline cudaError_t cudaFree(void* p) {
  std::free(p);
  return cudaSuccess;
}
inline cudaError_t cudaMemcpy(void* d, const void* s, size_t n, cudaMemcpyKind) {
  std::memmove(d, s, n);
  return cudaSuccess;
}
inline cudaError_t cudaMemcpyAsync(void* d, const void* s, size_t n, cudaMemcpyKind k, cudaStream_t = nullptr) {
  return cudaMemcpy(d, s, n, k);
}
inline cudaError_t cudaMemset(void* d, int v, size_t n) {
  std::memset(d, v, n);
  return cudaSuccess;
}
inline cudaError_t cudaMemsetAsync(void* d, int v, size_t n, cudaStream_t = nullptr) { return cudaMemset(d, v, n); }
inline cudaError_t cudaStreamSynchronize(cudaStream_t) { return cudaSuccess; }
inline cudaError_t cudaEventCreate(cudaEvent_t* e) {
  *e = reinterpret_cast<cudaEvent_t>(new char[1]);
  return cudaSuccess;
}
inline cudaError_t cudaEventDestroy(cudaEvent_t e) {
  delete[] reinterpret_cast<char*>(e);
  return cudaSuccess;
}
inline cudaError_t cudaEventRecord(cudaEvent_t, cudaStream_t = nullptr) { return cudaSuccess; }
inline cudaError_t cudaEventElapsedTime(float* ms, cudaEvent_t, cudaEvent_t) {
  *ms = 0.f;
  return cudaSuccess;
}
inline cudaError_t cudaGetDevice(int* d) {
  *d = 0;
  return cudaSuccess;
}
inline cudaError_t cudaDeviceGetAttribute(int* v, cudaDeviceAttr, int) {
  *v = 152;
  return cudaSuccess;
}
template <typename T>
inline cudaError_t cudaGetSymbolAddress(void** p, const T& symbol) {
  *p = const_cast<void*>(static_cast<const void*>(&symbol));
  return cudaSuccess;
}
