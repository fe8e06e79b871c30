// common.cuh -- shared pieces of the CUDA path: the device error word, the
// bounded pipeline wait, and the internal launcher declarations.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/attn.h"
#include "sm103_ptx.cuh"

namespace gb300 {

// Device error word layout: [0] = first error code, [1] = site id,
// [2] = blockIdx.x of the reporter, [3] = extra (iteration / value).
constexpr int kErrWords = 4;

// Wait budget for one pipeline wait: long enough to never fire on a healthy
// launch, short enough that a stuck pipeline returns within seconds.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// Site ids reported with ATTN_ERR_DEVICE_TIMEOUT.
enum WaitSite : int {
  kSiteQFull = 1,
  kSiteKvFull = 2,
  kSiteKvEmpty = 3,
  kSiteSFull = 4,
  kSitePFull = 5,
  kSitePvDone = 6,
  kSiteXchg = 7,
  kSiteXfree = 8,
  kSiteDrain = 9,
};

__device__ __forceinline__ void record_error(int* err, int code, int site, int extra) {
  if (err == nullptr) return;
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = site;
    err[2] = (int)blockIdx.x;
    err[3] = extra;
  }
}

// Bounded wait on an mbarrier phase.  Returns false (after recording
// ATTN_ERR_DEVICE_TIMEOUT and raising the CTA's abort flag) when the budget
// runs out, or immediately once another role of the CTA has aborted.
template <bool kClusterScope = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile int* abort_flag, int* err, int site,
                                          int extra) {
  auto probe = [&]() {
    return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  // A non-blocking test first: most waits find the phase complete already.
  if (!kClusterScope && mbar_test_wait(bar, parity)) return true;
  if (probe()) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (probe()) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
      *abort_flag = 1;
      record_error(err, ATTN_ERR_DEVICE_TIMEOUT, site, extra);
      return false;
    }
  }
}

}  // namespace gb300

// ---- internal launchers (C++ linkage, defined in the kernel files) ---------

struct PrefillF32Args {
  const float* q;
  const float* k;
  const float* v;
  float* o;
  float* lse;
  int B, H, N, D;
  int causal;
  float scale;
  int* err;
  int debug_skip_block;  // test hook: >=0 makes every CTA skip that K/V block's load
};

struct PrefillBf16Args {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, N, D;
  int causal;
  float scale;
  int* err;
  int num_sms;
  int debug_skip_load;  // test hook: >0 skips that K/V load (bounded-wait test)
};

struct PrefillTf32x3Args {
  const float* q;
  const float* k;
  const float* v;
  float* o;
  float* lse;
  int B, H, N, D;
  int causal;
  float scale;
  void* workspace;  // >= prefill_tf32x3_workspace_bytes(B, H, N)
  int* err;
  int debug_skip_block;  // test hook: >=0 makes every CTA skip that K/V block's load
};

struct MlaArgs {
  const void* q;
  const void* kv;
  const int32_t* block_table;
  const int32_t* seqlens;
  void* o;
  float* lse;
  int B, Hq;
  float scale;
  int max_blocks;
  int num_blocks;
  void* workspace;
  size_t workspace_bytes;
  int pages_per_split;
  int num_sms;
  int* err;
  int debug_skip_step;  // test hook: >=0 makes rank 1 of every cluster skip that step's load
};

// Each returns a cudaError_t (cudaSuccess on a clean enqueue) and may set a
// message through attn_set_error().
cudaError_t launch_prefill_f32(const PrefillF32Args& a, cudaStream_t s);
cudaError_t launch_prefill_bf16(const PrefillBf16Args& a, cudaStream_t s);
cudaError_t launch_mla_decode(const MlaArgs& a, cudaStream_t s);
cudaError_t launch_prefill_tf32x3(const PrefillTf32x3Args& a, cudaStream_t s);

// Kernel shape queries (host-only, no CUDA calls).
bool prefill_f32_info(int D, int* Br, int* Bc, int* threads, int* smem);
bool prefill_bf16_info(int D, int* Br, int* Bc, int* threads, int* smem);
size_t mla_workspace_bytes(int B, int Hq, int max_blocks, int num_sms, int pages_per_split);
size_t prefill_tf32x3_workspace_bytes(int B, int H, int N);
bool prefill_tf32x3_info(int* Br, int* Bc, int* threads, int* smem);

// Fixed-scratch support for mla_decode_noalloc (defined in mla_decode.cu).
cudaError_t mla_noalloc_scratch(void** ptr, size_t* bytes);
int mla_noalloc_max_batch();
int mla_noalloc_max_sms();

// Error-message helper shared by the host files.
void attn_set_error(const char* fmt, ...);
// The current device's error word (kernels record device-side failures in
// it); nullptr with *code_out set when it cannot be found.
int* attn_device_err_word(int* code_out);

// Driver entry point for cuTensorMapEncodeTiled (resolved once through cudart).
typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion,
                                    CUtensorMapFloatOOBfill);
PFN_encodeTiled get_encode_tiled();
