"""fp64 CPU oracle for multi-head latent attention (MLA) decode.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and
the CPU-baseline leg of the benchmark may import or call anything here.  The
product path (the CUDA library and its Python binding) never reaches this
package, and this package never imports the product: the two share no code.
The one module both consume is ``mla_inputs``, which draws the seeded inputs
and holds none of the method's arithmetic.

Everything is written from the definitions on the pages, plainly, in float64:

* "Multi-head latent attention (MLA)" (ai-knowledge-tree, pillar E3):
  section 2 (latent down-projection c_t = W^DKV h_t, up-projections W^UK,
  W^UV, folding them into the query/output), section 3 (decoupled RoPE key,
  score = content term + positional term), section 4 and Exercise 1 (cache
  numbers per token).
* "Attention, Part 2: MQA, GQA and MLA" (ishwarj.com): "The MLA equations",
  "The trick that makes it fast: never rebuild at all" (absorption of W_uk
  into the query, of W_uv after the latent-space value sum, the absorbed
  inference path and its causal mask), "Why position needs its own key"
  (RoPE pair rotation), "How big is the difference?" (cache sizes, 2.25
  groups).
* "How DeepSeek Rewrote the Transformer" (zhichai.net): absorbed
  projections, "V reused from K" (the value is the first d_c numbers of the
  cached row), the 56.9x estimate.

Parity status: every function in ``mla_oracle`` is pinned by a test in
``tests/test_oracle_pins.py`` against something other than itself (page
figures, a library attention routine, brute-force loops, closed forms and
invariants).  No function is "parity unpinned".
"""

from .mla_oracle import *  # noqa: F401,F403
