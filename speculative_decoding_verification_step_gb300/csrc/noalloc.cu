// Allocation-free variant of spec_accept_rows.
//
// Who needs it: callers that cannot allocate device memory at the moment
// they verify drafts.  A serving process that reserved (nearly) all of HBM
// up front for its own KV-cache pool has no room left for ad-hoc buffers,
// and a latency-critical decode loop cannot afford the implicit device-wide
// synchronisation that cudaMalloc / cudaFree may cause.  spec_accept_rows
// takes its scratch (per-chunk partials and per-row arrival tickets) from the
// stream-ordered allocator; this variant takes it from one fixed array
// compiled into the library instead and calls no allocating routine.
//
// The array (kNoAllocScratchBytes, 4 MiB) lives on every GPU that loads the
// library until the process exits.  All calls share it and it keeps the last
// call's contents: the tickets are cleared at the start of every call, the
// partials are always written before they are read.  Calls that overlap on
// the GPU (two streams, or two host threads without ordering) race on it.
#include <cuda_runtime.h>

#include <string>

#include "common.cuh"
#include "kernels.h"
#include "specverify.h"

namespace sv {
void set_thread_error(const std::string& msg);  // engine.cu
}

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_accept_scratch[kNoAllocScratchBytes];

// Device address of the array on the current device, looked up on every
// call (cheap; nothing cached, so a device reset that reloads the module
// leaves no stale address behind).
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_accept_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

int fail(int code, const std::string& msg) {
  sv::set_thread_error(msg);
  return code;
}

}  // namespace

extern "C" SPEC_API int spec_accept_rows_noalloc(
    const float* p_logits, int64_t p_row_stride, const float* q_logits, int64_t q_row_stride,
    const int32_t* drafts, int rows, int K, int V, float temperature, uint64_t seed,
    uint64_t step_base, int32_t* tokens, int32_t* counts, uint32_t* flags, void* stream) {
  if (!p_logits || !q_logits || !drafts || !tokens || !counts)
    return fail(SPEC_E_ARG, "spec_accept_rows_noalloc: null pointer");
  if (rows < 1 || K < 1 || K > 16 || V < 2 || !(temperature >= 0.f))
    return fail(SPEC_E_ARG, "spec_accept_rows_noalloc: bad size or temperature");
  if (rows > 65535) return fail(SPEC_E_ARG, "spec_accept_rows_noalloc: at most 65535 rows per call");
  const size_t pf = sv::accept_partial_floats(rows, K, V);
  const size_t partial_bytes = (pf * sizeof(float) + 255) & ~size_t(255);
  const size_t need = partial_bytes + (size_t)rows * sizeof(int);
  if (need > kNoAllocScratchBytes)
    return fail(SPEC_E_ARG, "spec_accept_rows_noalloc: needs " + std::to_string(need) +
                                " bytes of scratch, the fixed array holds " +
                                std::to_string(kNoAllocScratchBytes) +
                                " (use fewer rows per call or spec_accept_rows)");
  void* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess)
    return fail(SPEC_E_CUDA, std::string("spec_accept_rows_noalloc: cudaGetSymbolAddress: ") +
                                 cudaGetErrorString(e));
  cudaStream_t st = (cudaStream_t)stream;
  float* partials = (float*)base;
  int* tickets = (int*)((char*)base + partial_bytes);
  e = cudaMemsetAsync(tickets, 0, (size_t)rows * sizeof(int), st);
  if (e != cudaSuccess)
    return fail(SPEC_E_CUDA, std::string("spec_accept_rows_noalloc: ") + cudaGetErrorString(e));
  sv::AcceptDesc a{};
  a.p = p_logits; a.p_ld = p_row_stride; a.q = q_logits; a.q_ld = q_row_stride;
  a.drafts = drafts; a.rows = rows; a.K = K; a.V = V; a.temperature = temperature;
  a.seed = seed; a.step_base = step_base; a.out_tokens = tokens; a.out_count = counts;
  a.out_flags = flags; a.partials = partials; a.tickets = tickets;
  e = sv::launch_accept(a, st);
  if (e != cudaSuccess)
    return fail(SPEC_E_CUDA, std::string("spec_accept_rows_noalloc: ") + cudaGetErrorString(e));
  return SPEC_OK;
}
