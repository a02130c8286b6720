// fa_host.cu -- attention (forward and backward) from host buffers to host
// buffers, with the copies overlapped with the kernels.
//
// The batch is cut into chunks of whole batch entries (each [Bc][H][T][d]
// slice is contiguous in the [B][H][T][d] layout, and the batch entries are
// independent).  Chunk c runs on internal stream c % 2 through device slot
// c % 2 of the caller's workspace: copy in, kernels, copy out.  While one
// stream's kernels run, the other stream's copies proceed on the copy
// engines.  Reusing a slot waits for nothing extra: the chunk that last used
// it ran earlier on the same stream.  The two streams fork from the caller's
// stream and join back into it through events, so the call is asynchronous
// and can be captured in a CUDA graph.
#include <mutex>

#include "fa_internal.h"

namespace fa {

namespace {

// Two non-blocking streams and fork/join events per device, created on first
// use and kept for the life of the process.
struct HostPipes {
  cudaStream_t s[2] = {nullptr, nullptr};
  cudaEvent_t fork = nullptr, join[2] = {nullptr, nullptr};
  bool ready = false;
};
HostPipes g_pipes[64];
std::mutex g_pipes_mu;

// (called with g_pipes_mu held)
fa_status pipes_for_device(HostPipes** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
  HostPipes& p = g_pipes[dev];
  if (!p.ready) {
    for (int i = 0; i < 2; ++i) {
      if ((e = cudaStreamCreateWithFlags(&p.s[i], cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_status(e);
      if ((e = cudaEventCreateWithFlags(&p.join[i], cudaEventDisableTiming)) != cudaSuccess)
        return cuda_status(e);
    }
    if ((e = cudaEventCreateWithFlags(&p.fork, cudaEventDisableTiming)) != cudaSuccess)
      return cuda_status(e);
    p.ready = true;
  }
  *out = &p;
  return FA_OK;
}

struct ChunkSizes {
  int Bc;            // batch entries per chunk (the last may hold fewer)
  size_t q, kv, l;   // bytes per batch entry: Q (= O), K (= V), LSE
  size_t slot;       // bytes of one device slot (Q, K, V, O, LSE of a chunk)
};

size_t round16(size_t x) { return (x + 15) / 16 * 16; }

ChunkSizes chunk_sizes(int B, int Hq, int Hkv, int T, int d, fa_dtype dtype, int chunks) {
  ChunkSizes c;
  const size_t e = dtype == FA_DTYPE_F32 ? 4 : 2;
  c.Bc = (B + chunks - 1) / chunks;
  c.q = static_cast<size_t>(Hq) * T * d * e;
  c.kv = static_cast<size_t>(Hkv) * T * d * e;
  c.l = static_cast<size_t>(Hq) * T * 4;
  // Q, K, V, O, LSE of Bc entries, each region 16-byte aligned
  c.slot = 2 * round16(c.Bc * c.q) + 2 * round16(c.Bc * c.kv) + round16(c.Bc * c.l);
  return c;
}

}  // namespace

size_t host_workspace_bytes(int B, int Hq, int Hkv, int T, int d, fa_dtype dtype, int chunks) {
  return 2 * chunk_sizes(B, Hq, Hkv, T, d, dtype, chunks).slot;
}

fa_status run_fwd_host(const FwdArgs& a, int chunks, void* workspace) {
  // one enqueue sequence at a time: the streams and events are shared by
  // every call on the device (the GPU then runs overlapping calls in turn)
  std::lock_guard<std::mutex> lock(g_pipes_mu);
  HostPipes* p = nullptr;
  fa_status s = pipes_for_device(&p);
  if (s != FA_OK) return s;
  const ChunkSizes cs = chunk_sizes(a.B, a.Hq, a.Hkv, a.T, a.d, a.dtype, chunks);
  cudaError_t e = cudaEventRecord(p->fork, a.stream);
  if (e != cudaSuccess) return cuda_status(e);
  for (int i = 0; i < 2; ++i)
    if ((e = cudaStreamWaitEvent(p->s[i], p->fork, 0)) != cudaSuccess) return cuda_status(e);
  // on an error part of the chunks may already be enqueued: the streams still
  // join back into the caller's stream, so that synchronising it covers them
  fa_status result = FA_OK;
  for (int c = 0, b0 = 0; b0 < a.B && result == FA_OK; ++c, b0 += cs.Bc) {
    const int nb = a.B - b0 < cs.Bc ? a.B - b0 : cs.Bc;
    cudaStream_t st = p->s[c & 1];
    uint8_t* slot = static_cast<uint8_t*>(workspace) + (c & 1) * cs.slot;
    uint8_t* dq = slot;
    uint8_t* dk = dq + round16(cs.Bc * cs.q);
    uint8_t* dv = dk + round16(cs.Bc * cs.kv);
    uint8_t* dO = dv + round16(cs.Bc * cs.kv);
    float* dl = reinterpret_cast<float*>(dO + round16(cs.Bc * cs.q));
    const uint8_t* hq = static_cast<const uint8_t*>(a.q) + b0 * cs.q;
    const uint8_t* hk = static_cast<const uint8_t*>(a.k) + b0 * cs.kv;
    const uint8_t* hv = static_cast<const uint8_t*>(a.v) + b0 * cs.kv;
    if ((e = cudaMemcpyAsync(dq, hq, nb * cs.q, cudaMemcpyHostToDevice, st)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dk, hk, nb * cs.kv, cudaMemcpyHostToDevice, st)) != cudaSuccess ||
        (e = cudaMemcpyAsync(dv, hv, nb * cs.kv, cudaMemcpyHostToDevice, st)) != cudaSuccess) {
      result = cuda_status(e);
      break;
    }
    FwdArgs ca = a;
    ca.q = dq;
    ca.k = dk;
    ca.v = dv;
    ca.o = dO;
    ca.lse = dl;
    ca.B = nb;
    ca.stream = st;
    result = a.dtype == FA_DTYPE_F32 ? launch_simt(ca) : launch_tc(ca);
    if (result != FA_OK) break;
    uint8_t* ho = static_cast<uint8_t*>(a.o) + b0 * cs.q;
    uint8_t* hl = reinterpret_cast<uint8_t*>(a.lse) + b0 * cs.l;
    if ((e = cudaMemcpyAsync(ho, dO, nb * cs.q, cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
        (e = cudaMemcpyAsync(hl, dl, nb * cs.l, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
      result = cuda_status(e);
  }
  for (int i = 0; i < 2; ++i) {
    if ((e = cudaEventRecord(p->join[i], p->s[i])) != cudaSuccess ||
        (e = cudaStreamWaitEvent(a.stream, p->join[i], 0)) != cudaSuccess)
      if (result == FA_OK) result = cuda_status(e);
  }
  return result;
}

// ------------------------------------------------------------- backward
namespace {

struct BwdChunkSizes {
  int Bc;
  size_t q, kv, l;   // bytes per batch entry: Q (= O, dO, dQ), K (= V, dK, dV), LSE
  size_t rows;       // bytes of the backward's row workspace for Bc entries
  size_t slot;
};

BwdChunkSizes bwd_chunk_sizes(int B, int Hq, int Hkv, int T, int d, fa_dtype dtype, int chunks) {
  BwdChunkSizes c;
  const size_t e = dtype == FA_DTYPE_F32 ? 4 : 2;
  c.Bc = (B + chunks - 1) / chunks;
  c.q = static_cast<size_t>(Hq) * T * d * e;
  c.kv = static_cast<size_t>(Hkv) * T * d * e;
  c.l = static_cast<size_t>(Hq) * T * 4;
  c.rows = bwd_workspace_bytes(c.Bc, Hq, T);
  // Q, O, dO, dQ; K, V, dK, dV; LSE; rows
  c.slot = 4 * round16(c.Bc * c.q) + 4 * round16(c.Bc * c.kv) + round16(c.Bc * c.l) +
           round16(c.rows);
  return c;
}

}  // namespace

size_t bwd_host_workspace_bytes(int B, int Hq, int Hkv, int T, int d, fa_dtype dtype,
                                int chunks) {
  return 2 * bwd_chunk_sizes(B, Hq, Hkv, T, d, dtype, chunks).slot;
}

fa_status run_bwd_host(const BwdArgs& a, int chunks, void* workspace) {
  std::lock_guard<std::mutex> lock(g_pipes_mu);
  HostPipes* p = nullptr;
  fa_status s = pipes_for_device(&p);
  if (s != FA_OK) return s;
  const BwdChunkSizes cs = bwd_chunk_sizes(a.B, a.Hq, a.Hkv, a.T, a.d, a.dtype, chunks);
  cudaError_t e = cudaEventRecord(p->fork, a.stream);
  if (e != cudaSuccess) return cuda_status(e);
  for (int i = 0; i < 2; ++i)
    if ((e = cudaStreamWaitEvent(p->s[i], p->fork, 0)) != cudaSuccess) return cuda_status(e);
  fa_status result = FA_OK;
  for (int c = 0, b0 = 0; b0 < a.B && result == FA_OK; ++c, b0 += cs.Bc) {
    const int nb = a.B - b0 < cs.Bc ? a.B - b0 : cs.Bc;
    cudaStream_t st = p->s[c & 1];
    uint8_t* cur = static_cast<uint8_t*>(workspace) + (c & 1) * cs.slot;
    auto take = [&](size_t bytes) {
      uint8_t* r = cur;
      cur += round16(bytes);
      return r;
    };
    uint8_t* dq_in = take(cs.Bc * cs.q);   // Q
    uint8_t* d_o = take(cs.Bc * cs.q);     // O
    uint8_t* d_do = take(cs.Bc * cs.q);    // dO
    uint8_t* d_dq = take(cs.Bc * cs.q);    // dQ
    uint8_t* d_k = take(cs.Bc * cs.kv);
    uint8_t* d_v = take(cs.Bc * cs.kv);
    uint8_t* d_dk = take(cs.Bc * cs.kv);
    uint8_t* d_dv = take(cs.Bc * cs.kv);
    float* d_lse = reinterpret_cast<float*>(take(cs.Bc * cs.l));
    float* d_rows = reinterpret_cast<float*>(take(cs.rows));
    const size_t oq = b0 * cs.q, okv = b0 * cs.kv, ol = b0 * cs.l;
    struct In {
      void* dst;
      const void* src;
      size_t bytes;
    } ins[6] = {{dq_in, static_cast<const uint8_t*>(a.q) + oq, nb * cs.q},
                {d_k, static_cast<const uint8_t*>(a.k) + okv, nb * cs.kv},
                {d_v, static_cast<const uint8_t*>(a.v) + okv, nb * cs.kv},
                {d_o, static_cast<const uint8_t*>(a.o) + oq, nb * cs.q},
                {d_lse, reinterpret_cast<const uint8_t*>(a.lse) + ol, nb * cs.l},
                {d_do, static_cast<const uint8_t*>(a.d_o) + oq, nb * cs.q}};
    for (const In& in : ins)
      if ((e = cudaMemcpyAsync(in.dst, in.src, in.bytes, cudaMemcpyHostToDevice, st)) !=
          cudaSuccess) {
        result = cuda_status(e);
        break;
      }
    if (result != FA_OK) break;
    BwdArgs ca = a;
    ca.q = dq_in;
    ca.k = d_k;
    ca.v = d_v;
    ca.o = d_o;
    ca.lse = d_lse;
    ca.d_o = d_do;
    ca.dq = d_dq;
    ca.dk = d_dk;
    ca.dv = d_dv;
    ca.B = nb;
    ca.ws_delta = d_rows;
    ca.ws_lse2 = d_rows + static_cast<size_t>(nb) * a.Hq * bwd_rows_padded(a.T);
    ca.stream = st;
    result = launch_bwd_prep(ca);
    if (result == FA_OK) result = bwd_tc_supported(ca) ? launch_bwd_tc(ca) : launch_bwd_simt(ca);
    if (result != FA_OK) break;
    if ((e = cudaMemcpyAsync(static_cast<uint8_t*>(a.dq) + oq, d_dq, nb * cs.q,
                             cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
        (e = cudaMemcpyAsync(static_cast<uint8_t*>(a.dk) + okv, d_dk, nb * cs.kv,
                             cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
        (e = cudaMemcpyAsync(static_cast<uint8_t*>(a.dv) + okv, d_dv, nb * cs.kv,
                             cudaMemcpyDeviceToHost, st)) != cudaSuccess)
      result = cuda_status(e);
  }
  for (int i = 0; i < 2; ++i) {
    if ((e = cudaEventRecord(p->join[i], p->s[i])) != cudaSuccess ||
        (e = cudaStreamWaitEvent(a.stream, p->join[i], 0)) != cudaSuccess)
      if (result == FA_OK) result = cuda_status(e);
  }
  return result;
}

}  // namespace fa
