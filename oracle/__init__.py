"""CPU oracle for the write-time KV-cache path.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import anything from this
package.  The product library (``kv_cache_gb300``) never imports it, and this
package imports nothing from the product: the two share no code, tables or
constants.  Seeded input generation lives in ``kv_cache_gb300.synthetic``,
which holds none of the method's arithmetic; the oracle receives its inputs as
plain arrays.

What the oracle computes follows three public pages that report Runway's
real-time "Characters" serving work:

* [wechild] wechild.cn news item on Runway's real-time Characters inference
  paper (an untitled page; cited by paragraph).
* [neurocartel] neurocartel.com blog post "Runway Characters realtime on
  4 H100", section "Кэш: 240 attention calls и работа на запись".
* [ai.info] ai.info article "Characters funziona in tempo reale su quattro
  H100, afferma Runway", sections "La gestione della cache spostata al
  momento della scrittura" and "Latenza dei turni e altre configurazioni GPU".

Modules
-------
e4m3       FP8 e4m3fn codec written from the format's definition.
rope       1-D rotary position embedding with float64-reduced angles.
schemes    The naive scheme (shift, re-rotate and re-quantise the whole window
           on every call) and the write-time scheme (ring buffer, rotate and
           quantise once at write, one delta rotation per position reset).
attention  Softmax attention over the dequantised cache, in float64.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, library casts or brute force; none is "parity unpinned"
except that no page prints a tensor value, so no test compares the oracle
with a number printed on the pages (there is none to compare with).
"""
