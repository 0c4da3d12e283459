"""CPU oracle for the DSpark per-round draft -> schedule -> verify path.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, single-threaded numpy
restatement of what the DSpark pages define, written in float64 (the fp32 steps
are the ones the method itself fixes in fp32, each marked where it happens). It
exists to check the CUDA library and to serve as the timed CPU baseline. Only
the test suite, the smoke entry point and the benchmark's CPU-baseline /
reference arm may import it. The product path (the C-ABI library and its Python
binding) never imports, links or calls anything here, and this package never
imports the product path; the two share no code.

Sources (web pages about the paper "DSpark", cited by title and section):
  [GN]  "DSpark: Aceleração da inferência de LLM com speculative decoding [pdf]"
        (GeekNews, Portuguese summary) -- the densest technical source.
  [AI]  "DSpark: la apuesta de DeepSeek por la velocidad que no traiciona la
        calidad" (aitalk.it, Spanish essay).
  [JD]  "DeepSpec发布：让大模型生成提速6倍，输出质量却一点没变差" (jdon.com).

Modules:
  philox    counter-based uniforms U(seed, request, position, purpose)
  draft     Markov-head bias + tempered softmax + inverse-CDF draft sampling
  schedule  prefix-survival products + hardware-aware greedy prefix scheduler
  verify    lossless speculative-sampling verification (ratio test, residual,
            bonus token)
  round     the three stages chained, one request at a time

Parity status of each function is stated in its own docstring; the only
function without an independent pin is the residual/bonus sampler at full
vocabulary size (see verify.py), which is pinned only at small V by exact
enumeration and chi-square tests.
"""

from . import philox, draft, schedule, verify, round  # noqa: F401
