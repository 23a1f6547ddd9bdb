"""Plain, slow, obviously-correct CPU oracle for the paged KV-cache decode path.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute anything in this package. The only permitted callers are the test
suite (``tests/``), ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py``.

The oracle shares no code with the CUDA path: it does not import the
``paged_kv_cache_56_gb300`` package, and that package does not import this
one. The one thing both sides consume is the seeded synthetic input generator
(``paged_kv_cache_56_gb300.synth``), which holds none of the method's
arithmetic.

Sources (web pages, cited by title and section):

* [A] "无 vLLM 环境下的 Paged-KV 与连续批处理调度" (mixtureofinsights.com) --
  block pool of 16-token blocks (§1.2), KV-bytes formula (§2).
* [B] "vLLM核心概念：PagedAttention、Continuous Batching、KV Cache等原理"
  (5688vip.com, ch. 3) -- KV-cache size formula and 512 KB/token (§3.1),
  block tables and shared blocks (§3.2), A100 sizing (§3.5).
* [C] "离开 N 卡后的真实世界：Ultra x7 358h 平台上的 TTS 推理框架重构"
  (mixtureofinsights.com) -- FlashAttention tiling idea (§2), KV-bytes formula (§4).
* [D] "连续批处理与KV缓存" (5688vip.com, course ch. 4) -- free-block pool
  manager pseudocode (§4.2).
* [E] "轻量级推理引擎实战：KV Cache 量化与连续批处理的底层优化" (lpnh.cn) --
  decode reads the whole cache (§1), block table (§2.1), per-head symmetric
  INT8 quantizer and its dequantization (§3).

Modules:

* ``sizing``    -- closed-form KV-cache sizes and block counts.
* ``allocator`` -- FIFO free-block pool with per-request block lists.
* ``quantize``  -- symmetric INT8 block quantization (fp32, bit-exact target).
* ``attention`` -- single-token decode attention in fp64, and the merge of
  partial softmax states.
* ``cache``     -- contiguous per-sequence histories that quantize at their own
  fill points; produces the dequantized context a decode step attends over.
"""

from . import sizing, allocator, quantize, attention, cache  # noqa: F401
