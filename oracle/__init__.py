"""fp64 CPU oracle for the TokenGate gated-prefill path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.

Parity status per function (see the pins in ``tests/test_oracle_pins.py``):

* gate_score, gelu_erf    pinned (closed forms, library special cases)
* score_key, select_topk  pinned (brute-force rank definition, hand-worked fixture)
* logsigmoid, gather_rows pinned (closed forms, asymptotes, library routine)
* rmsnorm, qkv_proj       pinned (invariants, identity weight, brute-force loops)
* keybias_attn            pinned (SDPA special case, 2-key closed form, invariants)
* gated_layer, stack      composed of the pinned functions above
* keybias_attn_lse        pinned (q = 0 closed form, torch.logsumexp, row 0)
* keybias_attn_bias_grad,
  bias_grad_reduce        pinned (central differences of the forward, torch
                          SDPA autograd, 2-key closed form, shift invariance)
* attn_delta              pinned (brute-force loops, softmax written out)
* qk_rmsnorm, rope,
  swiglu_mlp              pinned (torch rms_norm / silu / linear; rope as a
                          complex rotation, identity at 0, norm and relative-
                          position invariance)
* qwen3_pruned_layer      pinned (reduces to the pinned stack layer and to the
                          identity; kept rows at original positions = the full
                          layer with pruned keys masked)
* the *learned* behaviour of a trained gate (which tokens it keeps on real
  text): parity unpinned, there are no trained weights or datasets here.
"""
from .tokengate_oracle import *  # noqa: F401,F403
from .tokengate_oracle import __all__  # noqa: F401
