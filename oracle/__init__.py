"""CPU oracle for training-free self-speculative decoding (CAS-Spec, CLaSp).

TEST INFRASTRUCTURE ONLY.  Only `tests/`, `__graft_entry__.smoke()` and the
`cpu_baseline` / `--impl reference` legs of `bench.py` may import or run
anything in this package.  The GPU library never calls it, and it shares no
code, table or constant generator with the GPU library: the two meet only in
`ssd_inputs` (seeded weights and prompts, no method arithmetic).

The oracle is the plain definition, written for a reader to check by eye:
numpy in float64, weights taken as the exact 16-bit values widened to
float64, one library matmul per projection, no fusion or blocking.  Two
decisions are taken in float32, the precision the GPU path takes them in:
the int8 quantization codes (quant.py) and greedy argmax / top-2 over the
logits (model.py).

Sources (web pages, cited by title and section):
  [CAS-blog]   "CAS-Spec技术：大型语言模型推理加速新方案" (intelliparadigm.com)
  [CAS-paper]  "CAS-Spec: Cascade Adaptive Self-Speculative Decoding for
               On-the-Fly Lossless Inference Acceleration of LLMs" (summary + abstract)
  [CLaSp]      CLaSp article (news.43b.com.cn/a/479818), sections 一..五

Modules:
  model.py    decoder forward (with early exit), KV cache, argmax/top-2,
              top-1 softmax probability
  quant.py    per-token int8 activation quantization
  decode.py   autoregressive greedy, linear (with draft exit) and tree
              speculative cycles, greedy acceptance + KV rollback, DyTC
              routing + EMA, horizontal and vertical cascade baselines
  clasp.py    CLaSp dynamic-programming skip search + brute force
  latency.py  latency model fit and cascade depth rules of the scheduler
"""
