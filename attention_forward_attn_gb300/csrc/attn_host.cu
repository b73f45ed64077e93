// attn_fwd_host: the forward with every buffer in host memory.
//
// The host link (about 0.2 TB/s each way on GB300, about 0.3 TB/s with both
// directions busy) is some thirty times slower than HBM, so a call that
// copies in, computes and copies out one after the other spends most of its
// time with the GPU idle.  Here the problem is cut into chunks of whole
// (batch, key/value head) slots -- each chunk a contiguous slice of Q, K, V,
// O and LSE -- and three queues overlap: host->device copies on one copy
// stream, the attention of each chunk on the caller's stream as soon as its
// inputs have landed, device->host copies of finished chunks on a second
// copy stream.  A call then takes about the time of its copies.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/attn.h"
#include "attn_internal.h"

namespace {

constexpr int kMaxDevices = 64;
// Input bytes of a full chunk: an eighth of the problem's input, kept within
// [8, 32] MiB, and larger only when that would make over 48 chunks.
constexpr int64_t kFullChunkMin = 8ll << 20;
constexpr int64_t kFullChunkMax = 32ll << 20;
constexpr int64_t kFullChunksPerProblem = 8;
constexpr int64_t kMaxChunks = 48;
constexpr int64_t kOneChunkBelow = 12ll << 20;  // smaller problems: one chunk

// Per-device streams of the host path and the events that order them: the
// caller's stream forks into them and joins them at the end.  One call
// queues at a time (mu), so reusing an event is safe: a cudaStreamWaitEvent
// waits for the record made before it was queued.
constexpr int kComputeStreams = 2;  // chunks alternate, so one chunk's tail overlaps the next

struct HostQueues {
  std::mutex mu;
  bool ready = false;
  cudaStream_t h2d = nullptr;                     // host -> device copies
  cudaStream_t conv = nullptr;                    // bf16: fp16 copies of newly landed V heads
  cudaStream_t comp[kComputeStreams] = {};        // attention calls
  cudaStream_t d2h = nullptr;                     // device -> host copies
  cudaEvent_t fork = nullptr;                     // caller's stream -> the streams above
  cudaEvent_t landed = nullptr;                   // a chunk's inputs are on the device
  cudaEvent_t converted = nullptr;                // ... and its V heads converted
  cudaEvent_t computed = nullptr;                 // a chunk's outputs are written
  cudaEvent_t joined[3 + kComputeStreams] = {};   // the streams above -> caller's stream

  cudaStream_t* streams[3 + kComputeStreams] = {&h2d, &conv, &comp[0], &comp[1], &d2h};
};

HostQueues g_queues[kMaxDevices];

void destroy_queues(HostQueues& hq) {
  for (cudaEvent_t* ev : {&hq.fork, &hq.landed, &hq.converted, &hq.computed}) {
    if (*ev != nullptr) cudaEventDestroy(*ev);
    *ev = nullptr;
  }
  for (cudaEvent_t& ev : hq.joined) {
    if (ev != nullptr) cudaEventDestroy(ev);
    ev = nullptr;
  }
  for (cudaStream_t* st : hq.streams) {
    if (*st != nullptr) cudaStreamDestroy(*st);  // released once its queued work finishes
    *st = nullptr;
  }
  hq.ready = false;
}

// Create the queues of the current device (caller holds hq.mu).
cudaError_t ensure_queues(HostQueues& hq) {
  if (hq.ready) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  for (cudaStream_t* st : hq.streams) {
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking);
  }
  for (cudaEvent_t* ev : {&hq.fork, &hq.landed, &hq.converted, &hq.computed}) {
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  }
  for (cudaEvent_t& ev : hq.joined) {
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {
    destroy_queues(hq);
    return e;
  }
  hq.ready = true;
  return cudaSuccess;
}

// One attention call of a chunk: B' batches x Hq' query heads over Hkv' K/V
// heads, starting at flattened query head q0 = b*Hq + h and K/V head kv0.
struct Piece {
  int64_t q0, kv0;
  int b, nb, hq, hkv;
};

// Cut the flattened query heads [u, u1) into calls whose head map is the
// plain h_kv = h_q / (Hq'/Hkv'): part of one group (Hkv' = 1), whole groups
// of one batch, or whole batches.  Calls f(piece) in order; returns the count.
template <class F>
int for_each_piece(int64_t u, int64_t u1, int Hq, int Hkv, F&& f) {
  const int group = Hq / Hkv;
  int n = 0;
  while (u < u1) {
    const int b = static_cast<int>(u / Hq), h = static_cast<int>(u % Hq);
    const int64_t rem = u1 - u;
    Piece pc;
    pc.q0 = u;
    pc.b = b;
    pc.kv0 = static_cast<int64_t>(b) * Hkv + h / group;
    if (h % group != 0 || rem < group) {
      pc.nb = 1;
      pc.hq = static_cast<int>(std::min<int64_t>(rem, group - h % group));
      pc.hkv = 1;
    } else if (h == 0 && rem >= Hq) {
      pc.nb = static_cast<int>(rem / Hq);
      pc.hq = Hq;
      pc.hkv = Hkv;
    } else {
      const int ng = static_cast<int>(std::min<int64_t>(rem / group, (Hq - h) / group));
      pc.nb = 1;
      pc.hq = ng * group;
      pc.hkv = ng;
    }
    f(pc);
    ++n;
    u += static_cast<int64_t>(pc.nb) * pc.hq;
  }
  return n;
}

// The chunk plan (validated sizes).  Chunks are ranges of flattened query
// heads; a chunk copies in its Q heads and the K/V heads that no earlier
// chunk copied.  Sizes ramp up from 1/8 of a full chunk (so the first kernel
// and the first device->host copy start early) and back down at the end (so
// little is left to compute and copy out after the last input lands).
// Returns the chunk count and writes the first min(count, cap) chunks.
int plan(int B, int Hq, int Hkv, int L, int D, attn_chunk_t* out, int cap) {
  const int64_t group = Hq / Hkv;
  const int64_t head = static_cast<int64_t>(L) * D * 2;
  const int64_t units = static_cast<int64_t>(B) * Hq;
  const int64_t total = static_cast<int64_t>(B) * (Hq + 2 * Hkv) * head;
  const int64_t full =
      std::max(std::min(std::max(total / kFullChunksPerProblem, kFullChunkMin), kFullChunkMax),
               (total + kMaxChunks - 1) / kMaxChunks);
  const int64_t first = full / 8;
  int n = 0;
  int64_t kv_done = 0;  // flattened K/V heads copied so far
  auto emit = [&](int64_t u0, int64_t u1, int64_t kv0, int64_t kv1) {
    if (n < cap) {
      out[n].q_head0 = static_cast<int>(u0);
      out[n].q_heads = static_cast<int>(u1 - u0);
      out[n].kv_head0 = static_cast<int>(kv0);
      out[n].kv_heads = static_cast<int>(kv1 - kv0);
      out[n].calls = for_each_piece(u0, u1, Hq, Hkv, [](const Piece&) {});
    }
    ++n;
  };
  if (total < kOneChunkBelow) {
    emit(0, units, 0, static_cast<int64_t>(B) * Hkv);
    return n;
  }
  int64_t u = 0, left = total;
  for (int c = 0; u < units; ++c) {
    const int64_t ramp = c < 3 ? first << c : full;
    const int64_t target = std::min(std::min(full, ramp), std::max(first, left / 2));
    int64_t end = u, bytes = 0, kv_seen = kv_done;
    while (end < units) {
      const int64_t kv = end / group;  // flattened K/V head of query head `end`
      const int64_t add = head + (kv >= kv_seen ? 2 * head : 0);
      if (end > u && bytes + add > target) break;
      bytes += add;
      if (kv >= kv_seen) kv_seen = kv + 1;
      ++end;
    }
    // a chunk of a whole group or more ends on a group boundary when that
    // drops at most a quarter of it: its calls are then whole groups (or
    // whole batches), not parts of a group
    if (end < units && end - u >= group && end % group != 0 && 4 * (end % group) <= end - u)
      end -= end % group;
    const int64_t kv0 = kv_done;
    kv_done = std::max(kv_done, (end - 1) / group + 1);
    left -= (end - u) * head + 2 * (kv_done - kv0) * head;
    emit(u, end, kv0, kv_done);
    u = end;
  }
  return n;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

namespace attn {

void host_path_shutdown() {
  int cur = 0;
  const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  for (int d = 0; d < kMaxDevices; ++d) {
    HostQueues& hq = g_queues[d];
    std::lock_guard<std::mutex> lock(hq.mu);
    if (!hq.ready) continue;
    if (cudaSetDevice(d) == cudaSuccess) destroy_queues(hq);
  }
  if (have_cur) cudaSetDevice(cur);
  cudaGetLastError();
}

}  // namespace attn

extern "C" {

attn_status_t attn_host_plan(int B, int Hq, int Hkv, int L, int D, attn_dtype_t dtype,
                             attn_chunk_t* chunks, int cap, int* n_chunks) {
  if (n_chunks == nullptr || cap < 0 || (cap > 0 && chunks == nullptr)) return ATTN_ERR_ARG;
  *n_chunks = 0;
  alignas(16) static unsigned char placeholder[16];  // stands in for the buffers in validate
  attn_status_t s = attn::validate(placeholder, placeholder, placeholder, placeholder, nullptr, B,
                                   Hq, Hkv, L, D, 1.f, 0, nullptr, dtype);
  if (s != ATTN_OK) return s;
  *n_chunks = plan(B, Hq, Hkv, L, D, chunks, cap);
  return ATTN_OK;
}

attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                            const int32_t* valid_len, attn_dtype_t dtype, attn_stream_t stream) {
  attn_status_t s = attn::validate(q, k, v, o, lse, B, Hq, Hkv, L, D, sm_scale, causal, valid_len,
                                   dtype);
  if (s == ATTN_ERR_ALIGN) s = ATTN_OK;  // host buffers: the copies need no alignment
  if (s != ATTN_OK) return s;
  int dev = 0, num_sms = 0;
  int* status_word = nullptr;
  if ((s = attn::current_device(&dev, &num_sms, &status_word)) != ATTN_OK) return s;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_ARCH;
  cudaMemPool_t pool = nullptr;
  if ((s = attn::device_pool(dev, &pool)) != ATTN_OK) return s;
  attn::TcConfig cfg;
  if (!attn::tc_config(D, &cfg)) return ATTN_ERR_HEADDIM;
  const bool bf16 = dtype == ATTN_BF16;

  std::vector<attn_chunk_t> chunks(static_cast<size_t>(plan(B, Hq, Hkv, L, D, nullptr, 0)));
  plan(B, Hq, Hkv, L, D, chunks.data(), static_cast<int>(chunks.size()));
  HostQueues& hq = g_queues[dev];
  std::lock_guard<std::mutex> lock(hq.mu);
  cudaError_t e = ensure_queues(hq);
  if (e != cudaSuccess) return attn::cuda_fail(e);

  // device copies of the whole problem in one allocation; bf16 adds the fp16
  // copy of V and its per-(K/V head, 128-key tile) flags
  const size_t head = static_cast<size_t>(L) * D * 2;  // bytes of one head's [L, D]
  const size_t n_kt = (static_cast<size_t>(L) + cfg.block_n - 1) / cfg.block_n;
  const size_t q_bytes = static_cast<size_t>(B) * Hq * head;
  const size_t kv_bytes = static_cast<size_t>(B) * Hkv * head;
  const size_t lse_bytes = lse != nullptr ? static_cast<size_t>(B) * Hq * L * 4 : 0;
  const size_t vl_bytes = valid_len != nullptr ? static_cast<size_t>(B) * 4 : 0;
  const size_t v16_bytes = bf16 ? kv_bytes : 0;
  const size_t flag_bytes = bf16 ? static_cast<size_t>(B) * Hkv * n_kt * 4 : 0;
  const size_t off_k = round256(q_bytes), off_v = off_k + round256(kv_bytes);
  const size_t off_o = off_v + round256(kv_bytes), off_lse = off_o + round256(q_bytes);
  const size_t off_vl = off_lse + round256(lse_bytes), off_v16 = off_vl + round256(vl_bytes);
  const size_t off_flags = off_v16 + round256(v16_bytes), total = off_flags + round256(flag_bytes);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* buf = nullptr;
  e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&buf), total, pool, cs);
  if (e != cudaSuccess) return attn::cuda_fail(e);
  uint8_t* d_q = buf;
  uint8_t* d_k = buf + off_k;
  uint8_t* d_v = buf + off_v;
  uint8_t* d_o = buf + off_o;
  float* d_lse = lse != nullptr ? reinterpret_cast<float*>(buf + off_lse) : nullptr;
  int32_t* d_vl = valid_len != nullptr ? reinterpret_cast<int32_t*>(buf + off_vl) : nullptr;
  uint8_t* d_v16 = bf16 ? buf + off_v16 : nullptr;
  int* d_flags = bf16 ? reinterpret_cast<int*>(buf + off_flags) : nullptr;
  const uint8_t* h_q = static_cast<const uint8_t*>(q);
  const uint8_t* h_k = static_cast<const uint8_t*>(k);
  const uint8_t* h_v = static_cast<const uint8_t*>(v);
  uint8_t* h_o = static_cast<uint8_t*>(o);

  attn_status_t result = ATTN_OK;
  auto step = [&](cudaError_t err) {
    if (err != cudaSuccess && result == ATTN_OK) result = attn::cuda_fail(err);
    return result == ATTN_OK;
  };
  auto status_step = [&](attn_status_t st) {
    if (st != ATTN_OK && result == ATTN_OK) result = st;
    return result == ATTN_OK;
  };
  // every stream of the host path starts after the work already on the caller's stream
  if (step(cudaEventRecord(hq.fork, cs))) {
    for (cudaStream_t* st : hq.streams) {
      if (!step(cudaStreamWaitEvent(*st, hq.fork, 0))) break;
    }
  }
  if (result == ATTN_OK && d_vl != nullptr) {
    step(cudaMemcpyAsync(d_vl, valid_len, vl_bytes, cudaMemcpyDefault, hq.h2d));
  }
  for (size_t c = 0; c < chunks.size() && result == ATTN_OK; ++c) {
    const attn_chunk_t ch = chunks[c];
    const size_t q0 = static_cast<size_t>(ch.q_head0), nq = static_cast<size_t>(ch.q_heads);
    const size_t kv0 = static_cast<size_t>(ch.kv_head0), nkv = static_cast<size_t>(ch.kv_heads);
    cudaStream_t comp = hq.comp[c % kComputeStreams];
    // inputs: the chunk's Q heads and the K/V heads no earlier chunk copied
    if (!step(cudaMemcpyAsync(d_q + q0 * head, h_q + q0 * head, nq * head, cudaMemcpyDefault,
                              hq.h2d)))
      break;
    if (nkv > 0 &&
        (!step(cudaMemcpyAsync(d_k + kv0 * head, h_k + kv0 * head, nkv * head, cudaMemcpyDefault,
                               hq.h2d)) ||
         !step(cudaMemcpyAsync(d_v + kv0 * head, h_v + kv0 * head, nkv * head, cudaMemcpyDefault,
                               hq.h2d))))
      break;
    if (!step(cudaEventRecord(hq.landed, hq.h2d)) || !step(cudaStreamWaitEvent(comp, hq.landed, 0)))
      break;
    if (bf16) {
      // fp16 copy of the new V heads on the conversion stream (in order, so
      // waiting for its latest record also covers every earlier chunk's heads)
      if (nkv > 0) {
        if (!step(cudaStreamWaitEvent(hq.conv, hq.landed, 0))) break;
        attn::Problem pv = attn::make_problem(nullptr, nullptr, d_v + kv0 * head, nullptr, nullptr,
                                              1, static_cast<int>(nkv), static_cast<int>(nkv), L,
                                              D, sm_scale, causal, nullptr, dtype,
                                              reinterpret_cast<attn_stream_t>(hq.conv),
                                              status_word);
        if (!step(attn::launch_vconv(pv, d_v16 + kv0 * head, d_flags + kv0 * n_kt)) ||
            !step(cudaEventRecord(hq.converted, hq.conv)))
          break;
      }
      if (!step(cudaStreamWaitEvent(comp, hq.converted, 0))) break;
    }
    // the attention calls of the chunk, cut at group and batch boundaries
    for_each_piece(static_cast<int64_t>(q0), static_cast<int64_t>(q0 + nq), Hq, Hkv,
                   [&](const Piece& pc) {
      if (result != ATTN_OK) return;
      const uint8_t* pq = d_q + pc.q0 * head;
      const uint8_t* pk = d_k + pc.kv0 * head;
      const uint8_t* pv = d_v + pc.kv0 * head;
      uint8_t* po = d_o + pc.q0 * head;
      attn::Problem p = attn::make_problem(
          pq, pk, pv, po, d_lse != nullptr ? d_lse + pc.q0 * L : nullptr, pc.nb, pc.hq, pc.hkv, L,
          D, sm_scale, causal, d_vl != nullptr ? d_vl + pc.b : nullptr, dtype,
          reinterpret_cast<attn_stream_t>(comp), status_word);
      CUtensorMap maps[5];
      if (!status_step(attn::encode_problem_maps(p, maps))) return;
      if (bf16 && !status_step(attn::encode_map(&maps[3], d_v16 + pc.kv0 * head, pc.nb, pc.hkv, L,
                                                D, attn::contiguous_strides(pc.hkv, L, D),
                                                cfg.block_n, false)))
        return;
      p.vflags = bf16 ? d_flags + pc.kv0 * n_kt : nullptr;
      step(attn::launch_tc(p, maps, num_sms));
    });
    if (result != ATTN_OK) break;
    // outputs of the chunk
    if (!step(cudaEventRecord(hq.computed, comp)) ||
        !step(cudaStreamWaitEvent(hq.d2h, hq.computed, 0)) ||
        !step(cudaMemcpyAsync(h_o + q0 * head, d_o + q0 * head, nq * head, cudaMemcpyDefault,
                              hq.d2h)))
      break;
    if (lse != nullptr) {
      step(cudaMemcpyAsync(lse + q0 * L, d_lse + q0 * L, nq * L * 4, cudaMemcpyDefault, hq.d2h));
    }
  }
  // join every stream into the caller's stream, then free (also after an
  // error, so that whatever was queued completes before the memory is reused)
  cudaError_t ej = cudaSuccess;
  for (int i = 0; i < 3 + kComputeStreams && ej == cudaSuccess; ++i) {
    ej = cudaEventRecord(hq.joined[i], *hq.streams[i]);
    if (ej == cudaSuccess) ej = cudaStreamWaitEvent(cs, hq.joined[i], 0);
  }
  if (ej != cudaSuccess) {
    // the caller's stream could not be ordered after them: wait for them here
    for (cudaStream_t* st : hq.streams) cudaStreamSynchronize(*st);
    step(ej);
  }
  step(cudaFreeAsync(buf, cs));
  return result;
}

}  // extern "C"
