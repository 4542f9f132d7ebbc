/* A decode step driven from plain C through the C ABI, with device buffers
 * from cudaMalloc and no other runtime: FULL summaries, score + Top-k + spans,
 * sparse decode over the paged cache. Built and run by
 * tests/test_gpu_c_consumer.py, which writes the inputs and checks the outputs
 * against the fp64 oracle.
 *
 * usage: gpu_c_consumer <in.bin> <out.bin>
 * in.bin:  int32 batch, n_qheads, n_kvheads, head_dim, block_size, max_blocks,
 *          k, n_pages; then q (bf16), kv_pages (bf16), block_table (int32),
 *          seq_lens (int32), in the layouts of include/kvsel.h.
 * out.bin: sel_idx (int32 [batch][k]), n_sel (int32 [batch]), out (fp32
 *          [batch][n_qheads][head_dim]), lse (fp32 [batch][n_qheads]). */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "kvsel.h"

static int fail(const char* what, int code) {
  fprintf(stderr, "%s failed: %d (%s)\n", what, code, kvsel_last_error());
  return 1;
}

static void* dev_alloc(size_t bytes) {
  void* p = NULL;
  if (cudaMalloc(&p, bytes ? bytes : 16) != cudaSuccess) return NULL;
  return p;
}

static int read_exact(FILE* f, void* dst, size_t bytes) { return fread(dst, 1, bytes, f) == bytes; }

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s in.bin out.bin\n", argv[0]);
    return 2;
  }
  FILE* fin = fopen(argv[1], "rb");
  if (!fin) return 2;
  int32_t hdr[8];
  if (!read_exact(fin, hdr, sizeof hdr)) return 2;
  kvsel_problem p = {hdr[0], hdr[1], hdr[2], hdr[3], hdr[4], hdr[5], hdr[6]};
  const int32_t k = hdr[6];
  const int64_t n_pages = hdr[7];
  const size_t q_n = (size_t)p.batch * p.n_qheads * p.head_dim;
  const size_t page_n = (size_t)p.n_kvheads * 2 * p.block_size * p.head_dim;
  const size_t kv_n = (size_t)n_pages * page_n;
  const size_t bt_n = (size_t)p.batch * p.max_blocks;
  kvsel_bf16* h_q = malloc(q_n * 2);
  kvsel_bf16* h_kv = malloc(kv_n * 2);
  int32_t* h_bt = malloc(bt_n * 4);
  int32_t* h_len = malloc((size_t)p.batch * 4);
  if (!h_q || !h_kv || !h_bt || !h_len) return 2;
  if (!read_exact(fin, h_q, q_n * 2) || !read_exact(fin, h_kv, kv_n * 2) ||
      !read_exact(fin, h_bt, bt_n * 4) || !read_exact(fin, h_len, (size_t)p.batch * 4))
    return 2;
  fclose(fin);

  cudaStream_t s;
  if (cudaStreamCreate(&s) != cudaSuccess) return 3;
  kvsel_bf16* q = dev_alloc(q_n * 2);
  kvsel_bf16* kv = dev_alloc(kv_n * 2);
  int32_t* bt = dev_alloc(bt_n * 4);
  int32_t* lens = dev_alloc((size_t)p.batch * 4);
  kvsel_bf16* summ = dev_alloc(bt_n * p.n_kvheads * p.head_dim * 2);
  double* acc = dev_alloc((size_t)p.batch * p.n_kvheads * p.head_dim * 8);
  int32_t* kps = dev_alloc((size_t)p.batch * 4);
  int32_t* sel = dev_alloc((size_t)p.batch * k * 4);
  int32_t* nsel = dev_alloc((size_t)p.batch * 4);
  int32_t* sst = dev_alloc((size_t)p.batch * k * 4);
  int32_t* sln = dev_alloc((size_t)p.batch * k * 4);
  int32_t* nsp = dev_alloc((size_t)p.batch * 4);
  uint8_t* dense = dev_alloc((size_t)p.batch);
  float* out = dev_alloc(q_n * 4);
  float* lse = dev_alloc((size_t)p.batch * p.n_qheads * 4);
  const size_t ws1n = kvsel_workspace_size(&p, KVSEL_WS_SCORE_TOPK);
  const size_t ws2n = kvsel_workspace_size(&p, KVSEL_WS_SPARSE_DECODE);
  void* ws1 = dev_alloc(ws1n);
  void* ws2 = dev_alloc(ws2n);
  if (!q || !kv || !bt || !lens || !summ || !acc || !kps || !sel || !nsel || !sst || !sln || !nsp ||
      !dense || !out || !lse || !ws1 || !ws2 || !ws1n || !ws2n)
    return 3;
  int32_t* h_k = malloc((size_t)p.batch * 4);
  for (int b = 0; b < p.batch; ++b) h_k[b] = k;
  cudaMemcpyAsync(q, h_q, q_n * 2, cudaMemcpyHostToDevice, s);
  cudaMemcpyAsync(kv, h_kv, kv_n * 2, cudaMemcpyHostToDevice, s);
  cudaMemcpyAsync(bt, h_bt, bt_n * 4, cudaMemcpyHostToDevice, s);
  cudaMemcpyAsync(lens, h_len, (size_t)p.batch * 4, cudaMemcpyHostToDevice, s);
  cudaMemcpyAsync(kps, h_k, (size_t)p.batch * 4, cudaMemcpyHostToDevice, s);
  cudaMemsetAsync(ws1, 0, ws1n, s);   /* workspaces start zero-filled */
  cudaMemsetAsync(ws2, 0, ws2n, s);
  kvsel_stream_t ks = (kvsel_stream_t)s;

  int r = kvsel_build_summaries(&p, KVSEL_SUMMARY_FULL, kv, n_pages, bt, lens, NULL, NULL, NULL, summ,
                                acc, ks);
  if (r) return fail("kvsel_build_summaries", r);
  r = kvsel_score_topk(&p, q, summ, lens, kps, 2.0f, 0.0f, sel, nsel, sst, sln, nsp, dense, NULL, ws1,
                       ws1n, ks);
  if (r) return fail("kvsel_score_topk", r);
  kvsel_kv_src src = {0};
  src.kind = KVSEL_KV_PAGED;
  src.kv_pages = kv;
  src.block_table = bt;
  src.n_pages = n_pages;
  const float scale = 1.0f / sqrtf((float)p.head_dim);
  r = kvsel_sparse_decode(&p, q, &src, lens, sel, nsel, sst, sln, nsp, dense, scale, out, NULL, lse,
                          ws2, ws2n, ks);
  if (r) return fail("kvsel_sparse_decode", r);
  r = kvsel_get_error(ks);   /* synchronises the stream */
  if (r) return fail("device error word", r);

  int32_t* h_sel = malloc((size_t)p.batch * k * 4);
  int32_t* h_nsel = malloc((size_t)p.batch * 4);
  float* h_out = malloc(q_n * 4);
  float* h_lse = malloc((size_t)p.batch * p.n_qheads * 4);
  cudaMemcpy(h_sel, sel, (size_t)p.batch * k * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(h_nsel, nsel, (size_t)p.batch * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(h_out, out, q_n * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(h_lse, lse, (size_t)p.batch * p.n_qheads * 4, cudaMemcpyDeviceToHost);
  if (cudaGetLastError() != cudaSuccess) return 3;
  FILE* fo = fopen(argv[2], "wb");
  if (!fo) return 2;
  fwrite(h_sel, 4, (size_t)p.batch * k, fo);
  fwrite(h_nsel, 4, (size_t)p.batch, fo);
  fwrite(h_out, 4, q_n, fo);
  fwrite(h_lse, 4, (size_t)p.batch * p.n_qheads, fo);
  fclose(fo);
  printf("c consumer ok\n");
  return 0;
}
