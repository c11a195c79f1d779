"""CPU oracle for the CSA2 attention step of DeepSeek-V4.1-Flash.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may use it.

It is a plain, slow, obviously correct restatement of what the step computes,
in numpy float64, written from the pages that describe the method:

* "DeepSeek V4.1-Flash. Every layer, connected" (sjtusm.pages.dev): "The query
  and output paths", "The global and index paths", and the hierarchical-indexer
  figure captions;
* "DeepSeek-V4.1-Flash explained" (snehal.ai): section 2 "CSA2", section 3
  "Hierarchical indexing", section 7 "FP4 global KV";
* the "deepseek-from-scratch" course (open-superintelligence-lab): the lessons
  "How CSA2 compresses, shares, and selects attention memory", "How DeepSeek
  stores its main KV cache in four-bit numbers", "05 / Sharing memory",
  "06 / Indexer and attention" and "07 / Hierarchical indexing";
* "DeepSeek V4 Inside" (blogs.gruheshkurra.com, the V4 predecessor, used only for
  mechanics the V4.1 pages also assert): "What does layer 0 sliding-window
  attention do to p?" (partial RoPE, the sink of eq. (27)) and "How does CSA
  compress 8 tokens into 4 KV entries?" (indexer scores, shared-KV MQA, output
  RoPE at -i).

It shares no code with the CUDA library and never imports it.  Every function
is pinned by a ``-m "not gpu"`` test in ``tests/test_oracle_pins.py`` against
values the pages print, closed forms, library routines or brute force; no
function here is "parity unpinned".
"""
from .csa2 import *  # noqa: F401,F403
from .writer import *  # noqa: F401,F403
from .compressor import *  # noqa: F401,F403
from .projections import *  # noqa: F401,F403
