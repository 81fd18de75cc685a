"""Plain CPU oracle for the speculative verify step.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
arm may use it. It shares no code with the CUDA path (no kernels, headers,
tables or helpers).

Everything is written from the definitions on the pages, in fp64 numpy unless
a page or a stated reading fixes another precision:

  attention.py  dense gather of the paged cache + textbook GQA attention with
                the offset causal mask ("KV Cache + Speculative Decoding",
                sections 5.3, 6.2, 6.3)
  sampling.py   scalar rejection sampler: accept test, residual resample,
                bonus token (quant67 "speculative decoding" section 3.1;
                "KV Cache + Speculative Decoding" sections 7.1-7.3, 7.6)
  kv_append.py  paged KV append ("KV Cache + Speculative Decoding" 6.2,
                append_token)
  fp8.py        OCP FP8 E4M3 encode/decode (used for the fp8 KV pools)
  theory.py     closed forms: alpha, residual mass, E[tau], speedup, KV bytes

Parity status: every function here is pinned by a -m "not gpu" test against
something other than itself (exact enumeration, closed forms, library
routines on special cases, Monte-Carlo laws, invariances). None is unpinned.
"""
from . import attention, fp8, kv_append, sampling, theory  # noqa: F401
