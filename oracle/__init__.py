"""Plain fp64 CPU oracle for sharded absorbed-MLA decode and its exact LSE merge.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code with the CUDA library under
``context_sharded_mla_gb300/``; the only module both sides use is the seeded
input generator in ``workloads/``, which holds none of the method's arithmetic.

The oracle is written from these pages (quoted by title and section):

* "Decode Context Parallelism" (zdszero.github.io/decode_context_parallelism):
  section "Core abstraction" (idea 1: ownership is a pure function of the
  slot, owner(p) = p mod N, row(p) = floor(p / N), chunk share
  count(a+L) - count(a); idea 2: each shard hands over (O_r, L_r)), section
  "Theory" (derivation of the merge identity, the merge operator and its
  numerically stable form, the base-e / base-2 pairing rule);
  section "通信策略" (the all-to-all and the AllGather + ReduceScatter merges);
  section "decode 路径：以 Kimi K3 的 MLA 为例" (w_kc / w_vc shapes).
* "MLA 的 Decode Context Parallelism" (ggaaooppeenngg.github.io): section 2
  (absorbed form: 576-d single-KV-head MQA, V = the 512-d c_K part, and the
  two absorption identities) and section 3 (the two-pass LSE merge).
* "PCP / DCP：计算、KV 布局与块轮转" (obnotes-4iw.pages.dev): section 5 (token
  round-robin), section 6 (block round-robin owner / local_index / local_len),
  section "KV cache 管理" (slot = page_id * page_size + offset).
* vLLM-Ascend "上下文并行（CP）" developer guide, section "块表" (virtual block
  slot mapping with cp_kv_cache_interleave_size).
* SGLang "Decode context parallelism" docs: sections "Virtual KV layout" and
  "MLA decode dataflow" (lse = logsumexp_r lse_r, o = sum_r exp(lse_r - lse) o_r).

Where the pages are silent or ambiguous the oracle takes one plain reading; each
reading is listed in the repository's design notes.

Modules
-------
``layout``      slot math, chunk share, vLLM virtual-block map, owner-filtered append.
``attention``   per-shard partial (o_r, lse_r), LSE merge, unsharded attention.
``bruteforce``  pure-Python loop versions for tiny inputs (pins for the above).
``absorb``      the query-side and output-side absorption products (identities 1, 2).
``exchange``    the cross-rank exchange of the partials: the all-to-all by head slice
                (and its wire format) and the AllGather + ReduceScatter merge.

Every function here is pinned by a ``-m "not gpu"`` test against the pages'
worked examples, closed forms, invariants or brute force.  None is unpinned.
"""

from . import layout, attention, bruteforce, absorb, exchange  # noqa: F401
