// ps_decode_graph.cu -- decode-step executor: one ps_decode_append captured once
// in a CUDA graph, stepped with its host copies in one call.
//
// A serving loop generates one token per step ("伪代码" section of the
// papers.ananclaw.com explainer): the new tokens' q, k, v and positions come
// from the host (sampling runs there) and the attention output goes back.
// Each step issues the same two kernels with the same parameters, so their
// host-side preparation (plan, tensor maps, RoPE table, launch attributes) is
// done once at capture; a step is then three stream operations -- copy in,
// graph launch, copy out -- issued back to back from native code, so the GPU
// does not sit idle between them waiting for the host.
#include <new>

#include "ps_internal.h"

namespace {

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

}  // namespace

struct ps_decode_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  void* inp = nullptr;
  void* res = nullptr;
  size_t in_bytes = 0, res_bytes = 0;
  int device = -1;
};

extern "C" ps_status_t ps_decode_step_layout_get(int32_t nseq, int32_t n_q_heads,
                                                 int32_t n_kv_heads, int32_t head_dim,
                                                 ps_decode_step_layout* L) {
  if (!L || nseq < 1 || n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads)
    return PS_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128) return PS_ERR_UNSUPPORTED;
  const size_t n = (size_t)nseq, D = (size_t)head_dim;
  L->q_off = 0;
  L->k_off = L->q_off + round256(n * n_q_heads * D * 2);
  L->v_off = L->k_off + round256(n * n_kv_heads * D * 2);
  L->pos_off = L->v_off + round256(n * n_kv_heads * D * 2);
  L->in_bytes = L->pos_off + round256(n * 4);
  L->out_off = 0;
  L->lse_off = round256(n * n_q_heads * D * 2);
  L->res_bytes = L->lse_off + round256(n * n_q_heads * 4);
  return PS_OK;
}

extern "C" ps_status_t ps_decode_graph_create(const ps_cache_desc* cache, int32_t n_q_heads,
                                              float scale, void* inp, void* res, void* workspace,
                                              size_t workspace_bytes, ps_decode_graph** out) {
  if (!out) return PS_ERR_INVALID_ARGUMENT;
  *out = nullptr;
  if (!cache || !inp || !res) return PS_ERR_INVALID_ARGUMENT;
  if (!aligned256(inp) || !aligned256(res)) return PS_ERR_ALIGNMENT;
  ps_decode_step_layout L;
  ps_status_t st = ps_decode_step_layout_get(cache->nseq, n_q_heads, cache->n_kv_heads,
                                             cache->head_dim, &L);
  if (st != PS_OK) return st;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return PS_ERR_CUDA;

  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return PS_ERR_CUDA;
  // Relaxed: the decode call sets kernel attributes and queries occupancy on the
  // host while it prepares its launches.
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    cudaStreamDestroy(s);
    return PS_ERR_CUDA;
  }
  uint8_t* in8 = static_cast<uint8_t*>(inp);
  uint8_t* res8 = static_cast<uint8_t*>(res);
  st = ps_decode_append(cache, in8 + L.q_off, in8 + L.k_off, in8 + L.v_off,
                        reinterpret_cast<const int32_t*>(in8 + L.pos_off), n_q_heads, scale,
                        res8 + L.out_off, reinterpret_cast<float*>(res8 + L.lse_off), workspace,
                        workspace_bytes, s);
  cudaGraph_t graph = nullptr;
  const cudaError_t end = cudaStreamEndCapture(s, &graph);  // always ends the capture
  cudaStreamDestroy(s);
  if (st == PS_OK && (end != cudaSuccess || !graph)) st = PS_ERR_CUDA;
  cudaGraphExec_t exec = nullptr;
  if (st == PS_OK && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) st = PS_ERR_CUDA;
  if (st != PS_OK) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();  // a failed capture leaves no sticky state behind
    return st;
  }
  ps_decode_graph* g = new (std::nothrow) ps_decode_graph;
  if (!g) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    return PS_ERR_CUDA;
  }
  g->graph = graph;
  g->exec = exec;
  g->inp = inp;
  g->res = res;
  g->in_bytes = L.in_bytes;
  g->res_bytes = L.res_bytes;
  g->device = device;
  *out = g;
  return PS_OK;
}

extern "C" ps_status_t ps_decode_graph_step(ps_decode_graph* g, const void* host_in,
                                            void* host_res, int32_t sync, void* stream) {
  if (!g) return PS_ERR_INVALID_ARGUMENT;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return PS_ERR_CUDA;
  if (device != g->device) return PS_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (host_in &&
      cudaMemcpyAsync(g->inp, host_in, g->in_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return PS_ERR_CUDA;
  if (cudaGraphLaunch(g->exec, s) != cudaSuccess) return PS_ERR_CUDA;
  if (host_res &&
      cudaMemcpyAsync(host_res, g->res, g->res_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PS_ERR_CUDA;
  if (sync && cudaStreamSynchronize(s) != cudaSuccess) return PS_ERR_CUDA;
  return PS_OK;
}

extern "C" ps_status_t ps_decode_graph_destroy(ps_decode_graph* g) {
  if (!g) return PS_OK;
  ps_status_t st = PS_OK;
  if (g->exec && cudaGraphExecDestroy(g->exec) != cudaSuccess) st = PS_ERR_CUDA;
  if (g->graph && cudaGraphDestroy(g->graph) != cudaSuccess) st = PS_ERR_CUDA;
  delete g;
  return st;
}
