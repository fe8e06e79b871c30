// host_path.cu -- the host-buffer entry points.  Inputs are copied in from
// host memory, the device path runs, and the results are copied back, all
// ordered on the caller's stream.  attn_fwd_host cuts the B*H heads into up
// to four contiguous chunks and overlaps them: while chunk c is computed on
// the caller's stream, chunk c+1 is copied in and chunk c-1 copied out on two
// copy streams of the library's own (one pair per device), with events for
// every hand-over and two device buffers used in turn.  mla_decode_host
// copies everything in, decodes and copies the result out in order (a block
// table may send any sequence to any page, so the pool is not chunked).
// No kernels live here.
#include <math.h>
#include <string.h>

#include <mutex>

#include "common.cuh"

namespace {

// Four chunks: the link moves ~210 GB/s host to device on one stream (a
// second adds nothing), so all but the last chunk's attention and copy-out
// hide under the copies in; eight chunks measured no better.
constexpr int kMaxChunks = 4;
constexpr int kMaxDev = 64;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// The copy streams and hand-over events of one device.  `mu` is held while
// one call enqueues: events are re-recorded by later calls, which is safe
// because every wait on them has been enqueued by then.
struct CopyStreams {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, up[2] = {}, done[2] = {}, down[2] = {};
  std::mutex mu;
  bool ready = false;
};
CopyStreams g_cs[kMaxDev];
std::mutex g_cs_mu;

cudaError_t copy_streams(CopyStreams** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_cs_mu);
  CopyStreams& c = g_cs[dev];
  if (!c.ready) {
    e = cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking);
    cudaEvent_t* evs[7] = {&c.start, &c.up[0], &c.up[1], &c.done[0], &c.done[1], &c.down[0],
                           &c.down[1]};
    for (int i = 0; i < 7 && e == cudaSuccess; ++i)
      e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
    c.ready = true;
  }
  *out = &c;
  return cudaSuccess;
}

// How attn_fwd_host cuts the work: `hc` heads per chunk, `nch` chunks, and
// one device buffer [q | k | v | o | lse] per chunk in flight.
struct HostPlan {
  int rows, hc, nch, esize;
  size_t tensor_bytes, lse_bytes, buf_bytes, total;
};

HostPlan host_plan(int B, int H, int N, int D, int dtype) {
  HostPlan p;
  p.esize = dtype == ATTN_DTYPE_F32 ? 4 : 2;
  p.rows = B * H;
  p.nch = p.rows < kMaxChunks ? p.rows : kMaxChunks;
  p.hc = (p.rows + p.nch - 1) / p.nch;
  p.nch = (p.rows + p.hc - 1) / p.hc;
  p.tensor_bytes = align256((size_t)p.hc * N * D * p.esize);
  p.lse_bytes = align256((size_t)p.hc * N * 4);
  p.buf_bytes = 4 * p.tensor_bytes + p.lse_bytes;
  p.total = (p.nch > 1 ? 2 : 1) * p.buf_bytes;
  return p;
}

bool host_args_ok(int B, int H, int N, int D, int dtype) {
  if (B <= 0 || H <= 0 || N <= 0 || D <= 0) return false;
  if ((long long)B * H * N > 0x7fffffffLL) return false;
  if (dtype == ATTN_DTYPE_F32) return D == 64;
  if (dtype == ATTN_DTYPE_BF16) return D == 64 || D == 128;
  return false;
}

struct MlaHostLayout {
  size_t q, kv, table, seqlens, o, lse, dec, total;
};

MlaHostLayout mla_host_layout(int B, int Hq, int max_blocks, int num_blocks, int num_sms) {
  MlaHostLayout w;
  size_t off = 0;
  w.q = off; off += align256((size_t)B * Hq * 576 * 2);
  w.kv = off; off += align256((size_t)num_blocks * 64 * 576 * 2);
  w.table = off; off += align256((size_t)B * max_blocks * 4);
  w.seqlens = off; off += align256((size_t)B * 4);
  w.o = off; off += align256((size_t)B * Hq * 512 * 2);
  w.lse = off; off += align256((size_t)B * Hq * 4);
  w.dec = off;
  off += align256(mla_workspace_bytes(B, Hq, max_blocks, num_sms, 0));
  w.total = off;
  return w;
}

int cuda_fail(cudaError_t e, const char* what) {
  attn_set_error("%s: %s", what, cudaGetErrorString(e));
  return ATTN_ERR_CUDA;
}

}  // namespace

extern "C" size_t attn_fwd_host_workspace_size(int B, int H, int N, int D, int dtype) {
  if (!host_args_ok(B, H, N, D, dtype)) return 0;
  return host_plan(B, H, N, D, dtype).total;
}

extern "C" int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int N, int D, int causal, float scale, int dtype,
                             void* workspace, size_t workspace_bytes, void* stream) {
  attn_set_error("%s", "");
  if (!q || !k || !v || !o || !lse || !workspace) {
    attn_set_error("attn_fwd_host: null pointer argument");
    return ATTN_ERR_INVALID_ARG;
  }
  if (B <= 0 || H <= 0 || N <= 0 || D <= 0 || !isfinite(scale)) {
    attn_set_error("attn_fwd_host: sizes must be >= 1 and scale finite");
    return ATTN_ERR_INVALID_ARG;
  }
  if (!host_args_ok(B, H, N, D, dtype)) {
    attn_set_error("attn_fwd_host: dtype %d with D=%d is not built (or B*H*N too large)",
                   dtype, D);
    return ATTN_ERR_UNSUPPORTED;
  }
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) {
    attn_set_error("attn_fwd_host: workspace must be 256-byte aligned");
    return ATTN_ERR_MISALIGNED;
  }
  const HostPlan p = host_plan(B, H, N, D, dtype);
  if (workspace_bytes < p.total) {
    attn_set_error("attn_fwd_host: workspace %zu < %zu bytes", workspace_bytes, p.total);
    return ATTN_ERR_WORKSPACE_TOO_SMALL;
  }
  CopyStreams* cs = nullptr;
  cudaError_t e = copy_streams(&cs);
  if (e != cudaSuccess) return cuda_fail(e, "attn_fwd_host: copy streams");
  std::lock_guard<std::mutex> lk(cs->mu);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t row_bytes = (size_t)N * D * p.esize;
  e = cudaEventRecord(cs->start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs->h2d, cs->start, 0);
  for (int c = 0; c < p.nch && e == cudaSuccess; ++c) {
    const int r0 = c * p.hc;
    const int nr = (p.rows - r0) < p.hc ? (p.rows - r0) : p.hc;
    const int b = c & 1;
    uint8_t* buf = ws + (size_t)b * p.buf_bytes;
    uint8_t* dq = buf;
    uint8_t* dk = buf + p.tensor_bytes;
    uint8_t* dv = buf + 2 * p.tensor_bytes;
    uint8_t* dout = buf + 3 * p.tensor_bytes;
    float* dl = reinterpret_cast<float*>(buf + 4 * p.tensor_bytes);
    const size_t off = (size_t)r0 * row_bytes, n = (size_t)nr * row_bytes;
    // buffer b was last used by chunk c-2: its results must be copied out
    if (c >= 2) e = cudaStreamWaitEvent(cs->h2d, cs->down[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dq, static_cast<const uint8_t*>(q) + off, n, cudaMemcpyHostToDevice,
                          cs->h2d);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dk, static_cast<const uint8_t*>(k) + off, n, cudaMemcpyHostToDevice,
                          cs->h2d);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(dv, static_cast<const uint8_t*>(v) + off, n, cudaMemcpyHostToDevice,
                          cs->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(cs->up[b], cs->h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, cs->up[b], 0);
    if (e != cudaSuccess) break;
    const int rc = attn_fwd(dq, dk, dv, dout, dl, 1, nr, N, D, causal, scale, dtype, s);
    if (rc != ATTN_OK) return rc;
    e = cudaEventRecord(cs->done[b], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs->d2h, cs->done[b], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<uint8_t*>(o) + off, dout, n, cudaMemcpyDeviceToHost,
                          cs->d2h);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(lse + (size_t)r0 * N, dl, (size_t)nr * N * 4, cudaMemcpyDeviceToHost,
                          cs->d2h);
    if (e == cudaSuccess) e = cudaEventRecord(cs->down[b], cs->d2h);
  }
  // the copy stream runs in order: its last copy-out covers every earlier one
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, cs->down[(p.nch - 1) & 1], 0);
  if (e != cudaSuccess) return cuda_fail(e, "attn_fwd_host: enqueue");
  return ATTN_OK;
}

extern "C" size_t mla_decode_host_workspace_size(int B, int Hq, int max_blocks_per_seq,
                                                 int num_blocks, int num_sms) {
  if (B <= 0 || Hq != 128 || max_blocks_per_seq <= 0 || num_blocks <= 0 || num_sms < 2)
    return 0;
  return mla_host_layout(B, Hq, max_blocks_per_seq, num_blocks, num_sms).total;
}

extern "C" int mla_decode_host(const void* q, const void* kv_cache, const int32_t* block_table,
                               const int32_t* seqlens, void* o, float* lse, int B, int Hq,
                               float scale, int max_blocks_per_seq, int num_blocks,
                               void* workspace, size_t workspace_bytes, void* stream) {
  attn_set_error("%s", "");
  if (!q || !kv_cache || !block_table || !seqlens || !o || !lse || !workspace) {
    attn_set_error("mla_decode_host: null pointer argument");
    return ATTN_ERR_INVALID_ARG;
  }
  if (B <= 0 || Hq <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || !isfinite(scale)) {
    attn_set_error("mla_decode_host: sizes must be >= 1 and scale finite");
    return ATTN_ERR_INVALID_ARG;
  }
  if (Hq != 128) {
    attn_set_error("mla_decode_host: built for Hq=128 (got %d)", Hq);
    return ATTN_ERR_UNSUPPORTED;
  }
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) {
    attn_set_error("mla_decode_host: workspace must be 256-byte aligned");
    return ATTN_ERR_MISALIGNED;
  }
  int dev = 0, nsm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "mla_decode_host: device query");
  const MlaHostLayout w = mla_host_layout(B, Hq, max_blocks_per_seq, num_blocks, nsm);
  if (workspace_bytes < w.total) {
    attn_set_error("mla_decode_host: workspace %zu < %zu bytes", workspace_bytes, w.total);
    return ATTN_ERR_WORKSPACE_TOO_SMALL;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t qb = (size_t)B * Hq * 576 * 2, kvb = (size_t)num_blocks * 64 * 576 * 2;
  const size_t tb = (size_t)B * max_blocks_per_seq * 4, sb = (size_t)B * 4;
  e = cudaMemcpyAsync(ws + w.q, q, qb, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ws + w.kv, kv_cache, kvb, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ws + w.table, block_table, tb, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ws + w.seqlens, seqlens, sb, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "mla_decode_host: copy in");
  const int rc = mla_decode(ws + w.q, ws + w.kv, reinterpret_cast<const int32_t*>(ws + w.table),
                            reinterpret_cast<const int32_t*>(ws + w.seqlens), ws + w.o,
                            reinterpret_cast<float*>(ws + w.lse), B, Hq, scale,
                            max_blocks_per_seq, num_blocks, ws + w.dec, w.total - w.dec, s);
  if (rc != ATTN_OK) return rc;
  e = cudaMemcpyAsync(o, ws + w.o, (size_t)B * Hq * 512 * 2, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(lse, ws + w.lse, (size_t)B * Hq * 4, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "mla_decode_host: copy out");
  return ATTN_OK;
}
