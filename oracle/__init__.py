"""CPU oracle for jagged softmax attention and its host tile scheduler.

TEST INFRASTRUCTURE. Only the tests, the smoke check of ``__graft_entry__``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may
import anything from this package. The product path (the CUDA library and its
Python binding) never imports, links or calls it, and the oracle imports
nothing from the product.

Sources followed (web pages on Jagged Flash Attention):

* "Desarrollo de Jagged Flash Attention para el modelo GEM"
  (noticiasdeia.es, Meta JFA / TLX / NVIDIA Blackwell article), cited below
  as [JFA-GEM]: packed Q/K/V with an offsets tensor, exact FlashAttention on
  it, the host LPT + zigzag tile scheduler, broadcast-Q with a summed dQ.
* "TLX Block Attention: a warp-specialized Blackwell kernel for fixed
  block-sparse ..." (noticias.mechatronicstore.cl), cited as [TLX-BA]: the
  standard FlashAttention inner loop and its stored log-sum-exp (section 2),
  Di = rowsum(dO * O) (section 2 and section 4), block-diagonal attention
  on fixed 64-token blocks (sections 1-2).
* "A PyTorch TLX-kernellel gyorsította a Meta hirdetési modelljének
  figyelmét" (aihirek.info), cited as [PT-TLX]: same method, summarised.

Modules:

* :mod:`oracle.attention` -- fp64 NumPy attention, forward and backward,
  for the jagged, broadcast-Q and block-diagonal layouts.
* :mod:`oracle.sched` -- plain-Python LPT sort and zigzag deal of tiles to SMs.

Every function here is pinned by a ``-m "not gpu"`` test in ``tests/``
against something other than itself (closed forms, a library routine,
finite differences, brute force); none is "parity unpinned".
"""
